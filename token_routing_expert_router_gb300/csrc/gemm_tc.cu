// The grouped expert GEMMs and the router GEMM on the 5th-generation tensor cores.
//
// "Grouped GEMM" runs all experts' GEMMs in one kernel to fill the tensor cores, and the
// kernels read the dynamic per-expert shapes from device memory instead of synchronising
// with the host ("Scalable Training of Mixture-of-Experts Models with Megatron Core"
// summary, section 2.4). Here that is one persistent kernel per GEMM:
//   * warp 0: TMA producer (128-byte-swizzled K-major tiles into a ring of smem stages);
//   * warp 1: TMEM owner and the single thread issuing tcgen05.mma (M = 128, N = BN);
//   * warps 2-5: epilogue, one TMEM lane (= one output row) per thread, two TMEM
//     accumulators so a tile's epilogue overlaps the next tile's main loop.
// Tiles are ordered group-major, then N tile, then M tile (fastest), so CTAs running at the
// same time share each weight tile through L2 and empty groups produce no tiles; a hot
// group's many M tiles spread over every SM. Ragged segment tails are handled by loading
// the full 128-row box (rows past the segment belong to the next group or are zero-filled
// past the end of the tensor) and storing only the segment's rows.
// CTA pairs of the forward GEMMs run a tile holding at most 64 of a segment's rows
// (its tail) with the operands swapped: the MMA's M side is the tile's 256 weight rows and
// its N side the tail's tokens rounded up to 32, so the tile costs the tensor core N / 256
// of a full one. It follows the segment's full tiles of the same weight block, which read
// that block from HBM at about the same time, so its weight loads mostly hit L2.
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "tc_common.cuh"

namespace moe {
namespace tc {
namespace {

constexpr int BM = 128;            // rows per tile (TMEM lanes)
constexpr int BK = 64;             // bf16 K per stage: one 128-byte swizzle row
constexpr int kThreads = 192;      // 6 warps
constexpr int kMaxGroups = 514;    // routed experts (<= 512) + one extra group + 1
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s: no legitimate wait comes close
constexpr int kSwapRows = 64;      // CTA pairs: tails of at most this many rows go tokens-on-N

// EPI_STORE_GU: the gate/up GEMM (B = gate and up rows, as for SwiGLU) storing g and u
// themselves, for the backward's recomputation of the activation. EPI_SWIGLU_GU: the
// forward's SwiGLU epilogue that also keeps g and u (out2), so that the backward recomputes
// only the activation and not this GEMM.
// EPI_SWIGLU_GATHER: EPI_SWIGLU_BF16 for single CTAs whose A rows are gathered by token with
// cp.async (its own instantiation, so the plain GEMM1 does not carry the gather's registers).
enum Epi {
  EPI_SWIGLU_BF16 = 0,
  EPI_STORE_BF16 = 1,
  EPI_STORE_F32_BIAS = 2,
  EPI_STORE_GU = 3,
  EPI_SWIGLU_GU = 4,
  EPI_SWIGLU_GATHER = 5
};

struct TcParams {
  const int32_t* offsets;   // [G+1] routed segment starts (device); may be null when G = 0
  int G;                    // routed groups
  int has_extra;            // one more group of T_extra rows (shared expert, or the router's
  int T_extra;              //   single problem), A from tmA2 at row a2_row_base
  int a2_row_base;
  int64_t out_extra_base;   // output row of the extra group's row 0
  int K;                    // reduction length, multiple of BK
  int n_tiles;              // N tiles per group
  int b_group_rows;         // rows of B per routed group
  int ldc;                  // output row length in elements
  void* out;
  void* out2;               // EPI_SWIGLU_GU: g and u [rows, ldc2] in 128-column blocks (g, then u)
  int ldc2;
  const float* bias;        // EPI_STORE_F32_BIAS: [N] or null
  const int32_t* row_token; // non-null: routed A rows are gathered, row r = token row_token[r]
                            //   of tmA (a one-row-box map of x); else tmA holds the rows
  const uint8_t* a_rows;    // with row_token on single CTAs: x itself (rows copied by cp.async)
  int64_t a_ld_bytes;       //   and its row length in bytes
  // EPI_STORE_BF16 with w_topk non-null: routed row r is scaled by its routing weight
  // w_topk[t * w_k + j] before rounding, t = w_row_token[r] and j the slot with
  // w_tok_row[t * w_k + j] == r (the routing weight applied in the down projection's epilogue)
  const int32_t* w_row_token;
  const int32_t* w_tok_row;
  const float* w_topk;
  int w_k;
  int swap_rows;            // CTA pairs, plain GEMM1 / GEMM2: tiles of at most this many rows
                            //   run with tokens on the MMA's N axis (0: never)
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// The tokens-on-N tail tiles' own boxes: A rows 16 at a time (routed and extra group) and,
// for GEMM1, 64-row boxes of the gate and up weights, so that each CTA holds the gate and
// up rows of the same 64 features.
struct SwapMaps {
  CUtensorMap t16, t16x, g64, u64, g64x, u64x;
};

// Named barrier 2 over the four epilogue warps (the tail tiles' gate/up exchange).
__device__ __forceinline__ void swap_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Shared memory of one CTA. CG = 2 (a CTA pair) halves the B rows each CTA holds, so a
// stage is 32 KB instead of 48 KB and six stages fit instead of four.
template <int BN, int CG>
struct Smem {
  static constexpr int kABytes = BM * BK * 2;                // 16 KB
  static constexpr int kBBytes = (BN / CG) * BK * 2;         // this CTA's B rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kStageBytes > 32768 ? 4 : 6;
  static constexpr int kTmemCols = 2 * BN;                   // two accumulators
  static constexpr size_t kBytes = 1024 /*align slack*/ + (size_t)kStages * kStageBytes + 256 /*barriers*/ +
                                   2 * kMaxGroups * sizeof(int32_t) + 4 * 2048 /*epilogue store staging*/;
};

// CG = 1: one CTA per 128-row tile (tcgen05.mma.cta_group::1, M = 128).
// CG = 2: a cluster of two CTAs per 256-row tile (cta_group::2, M = 256): each CTA loads its
// 128 A rows and half of the tile's B rows (SwiGLU: CTA 0 the gate rows, CTA 1 the up rows);
// the leader (rank 0) waits for both halves on its own barrier, issues the MMAs, and its
// commits arrive on both CTAs' barriers; each CTA's epilogue drains its own TMEM rows and
// the second CTA's epilogue reports to the leader's barrier.
template <int BN, int EPI, int CG>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmB0x, const __grid_constant__ CUtensorMap tmB1x,
                        const __grid_constant__ SwapMaps sw, const TcParams p) {
  using S = Smem<BN, CG>;
  constexpr int STAGES = S::kStages;
  constexpr int TM = BM * CG;  // rows of an m tile
  constexpr bool kSwiGLU = EPI == EPI_SWIGLU_BF16 || EPI == EPI_SWIGLU_GU;
  constexpr bool kSwapTail = CG == 2 && BN == 256 && (kSwiGLU || EPI == EPI_STORE_BF16);
  // a tail tile: its tokens (rounded up to 32) on the MMA's N axis
  auto swap_tile = [&](int rows) { return kSwapTail && rows <= p.swap_rows; };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * S::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * S::kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(bars + 32);  // [ngroups + 1]
  int32_t* seg_rows = mt_prefix + kMaxGroups;                 // [ngroups]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.G + p.has_extra;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG, nunits = gridDim.x / CG;  // tile walkers (CTAs or pairs)

  // ---- per-block setup: barriers, TMEM, and the m-tile prefix over the groups
  // single CTAs gather A rows with cp.async: each stage's barrier then also takes one
  // arrival per producer lane (after its copies are complete and fenced to the async proxy)
  const bool lsu_gather = CG == 1 && EPI == EPI_SWIGLU_GATHER && p.row_token != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], lsu_gather ? 33 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * CG);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (EPI == EPI_SWIGLU_BF16 || EPI == EPI_STORE_GU || EPI == EPI_SWIGLU_GU || EPI == EPI_SWIGLU_GATHER)
      tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) tmem_alloc_cg<CG>(tmem_slot, S::kTmemCols);
  if (warp == 2) build_tile_prefix(p.offsets, p.G, ngroups, p.T_extra, TM, lane, seg_rows, mt_prefix);
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.n_tiles * mt_prefix[ngroups];
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ======================= TMA producer (every CTA loads its own halves). Lane 0 issues
    // the box loads; with gathered A rows every lane gathers four of the 128 rows.
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool ok = true;
    // cp.async stages whose arrival is still owed: the npend fills starting at slot pend0
    // (consecutive), at most kPend of them, so a slot is always refilled after its arrival
    constexpr int kPend = 2;
    int pend0 = 0, npend = 0;
    auto arrive_oldest = [&]() {
      fence_proxy_async_smem();
      mbar_arrive(&full[pend0]);
      pend0 = pend0 + 1 == STAGES ? 0 : pend0 + 1;
      --npend;
    };
    auto drain_pending = [&]() {
      if (npend > 0) {
        cp_async_wait<0>();
        while (npend > 0) arrive_oldest();
      }
    };
    for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
      const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
      const bool extra = c.g >= p.G;
      const bool gather = p.row_token != nullptr && !extra;
      if (lsu_gather && !gather) drain_pending();
      const CUtensorMap* ta = extra ? &tmA2 : &tmA;
      const CUtensorMap* tb0 = extra ? &tmB0x : &tmB0;
      const CUtensorMap* tb1 = extra ? &tmB1x : &tmB1;
      const int a_row = (extra ? p.a2_row_base : p.offsets[c.g]) + c.mb * TM + (int)rank * BM;
      constexpr bool kGatedB =
          EPI == EPI_SWIGLU_BF16 || EPI == EPI_STORE_GU || EPI == EPI_SWIGLU_GU ||
          EPI == EPI_SWIGLU_GATHER;  // B = gate + up rows
      const int b_tile_rows = kGatedB ? BN / 2 : BN;  // rows of B per N tile
      int b_row = (extra ? 0 : c.g * p.b_group_rows) + c.nb * b_tile_rows;
      if (CG == 2 && !kGatedB) b_row += (int)rank * (BN / 2);
      const CUtensorMap* tb_mine = (CG == 2 && kGatedB && rank == 1) ? tb1 : tb0;
      int tok[4] = {0, 0, 0, 0};
      // single CTAs (only GEMM1 gathers): the token of row 4 i + lane / 8, i < 32
      constexpr bool kLsuRows = CG == 1 && EPI == EPI_SWIGLU_GATHER;
      int tokrow[kLsuRows ? 32 : 1];
      if (gather) {  // tokens of this lane's rows; rows past the segment repeat its last row
        const int seg_end = p.offsets[c.g + 1];
        if constexpr (kLsuRows) {
#pragma unroll
          for (int i = 0; i < 32; ++i) tokrow[i] = p.row_token[min(a_row + 4 * i + (lane >> 3), seg_end - 1)];
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) tok[i] = p.row_token[min(a_row + 4 * lane + i, seg_end - 1)];
        }
      }
      for (int kb = 0; kb < kblocks; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, abort, p.timeout_ns, p.status));
        if (!ok) break;
        uint8_t* a_dst = sA + stage * S::kABytes;
        uint8_t* b_dst = sB + stage * S::kBBytes;
        if constexpr (CG == 1) {
          if (lane == 0) mbar_arrive_expect_tx(&full[stage], gather ? S::kBBytes : S::kStageBytes);
          if (kLsuRows && gather) {
            // 128 rows x 8 16-byte pieces; 8 consecutive lanes take one row's 128 bytes, so a
            // warp instruction moves 4 whole rows (4 lines), into the 128-byte swizzle a TMA
            // box load writes (piece q of row r at r * 128 + 16 * (q ^ (r % 8)))
            const uint32_t a_base = smem_addr(a_dst);
            const int q = lane & 7, rsub = lane >> 3;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int r = 4 * i + rsub;
              cp_async16(a_base + r * 128 + 16 * (q ^ (r & 7)),
                         p.a_rows + (int64_t)tokrow[i] * p.a_ld_bytes + (int64_t)kb * BK * 2 + 16 * q);
            }
            cp_async_commit();
            if (npend == 0) pend0 = stage;
            ++npend;
            if (npend > kPend) {  // the oldest stage's copies are done: fence and arrive
              cp_async_wait<kPend>();
              arrive_oldest();
            }
          } else {
            if (lane == 0) tma_load_2d(ta, a_dst, &full[stage], kb * BK, a_row);
            if (lsu_gather) mbar_arrive(&full[stage]);  // the lanes' share of the count
          }
          if (lane == 0) {
            if (kGatedB) {
              tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);                    // gate rows
              tma_load_2d(tb1, b_dst + (BN / 2) * BK * 2, &full[stage], kb * BK, b_row);  // up rows
            } else {
              tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);
            }
          }
        } else if (swap_tile(c.rows)) {
          // tail tile: this CTA's 128 weight rows into the A slot (GEMM1: 64 gate + 64 up rows
          // of features [128 nb + 64 rank, +64); GEMM2: its usual 128 rows) and its half of
          // the tokens (16 or 32 rows) into the B slot
          const int nhalf = ((c.rows + 31) & ~31) / 2;
          if (lane == 0) {
            if (leader) mbar_arrive_expect_tx(&full[stage], 2u * (uint32_t)(S::kABytes + nhalf * BK * 2));
            const uint32_t bar = mapa_shared(smem_addr(&full[stage]), 0);
            if (kGatedB) {
              const int wrow = (extra ? 0 : c.g * p.b_group_rows) + c.nb * b_tile_rows + (int)rank * 64;
              tma_load_2d_pair(extra ? &sw.g64x : &sw.g64, a_dst, bar, kb * BK, wrow);
              tma_load_2d_pair(extra ? &sw.u64x : &sw.u64, a_dst + 64 * BK * 2, bar, kb * BK, wrow);
            } else {
              tma_load_2d_pair(tb0, a_dst, bar, kb * BK, b_row);
            }
            const int trow = (extra ? p.a2_row_base : p.offsets[c.g]) + c.mb * TM + (int)rank * nhalf;
            for (int j = 0; j < nhalf; j += 16)
              tma_load_2d_pair(extra ? &sw.t16x : &sw.t16, b_dst + j * BK * 2, bar, kb * BK, trow + j);
          }
        } else {
          // both CTAs' loads complete on the leader's barrier, which expects both
          if (lane == 0 && leader) mbar_arrive_expect_tx(&full[stage], 2 * S::kStageBytes);
          const uint32_t bar = mapa_shared(smem_addr(&full[stage]), 0);
          if (gather) {
            tma_gather4_pair(ta, a_dst + lane * 4 * BK * 2, bar, kb * BK, tok[0], tok[1], tok[2], tok[3]);
          } else if (lane == 0) {
            tma_load_2d_pair(ta, a_dst, bar, kb * BK, a_row);
          }
          if (lane == 0) tma_load_2d_pair(tb_mine, b_dst, bar, kb * BK, b_row);
        }
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    drain_pending();
    if (lane == 0) {
      // tail: every stage's last fill has been consumed (so no TMA write or MMA commit
      // is still in flight when the block exits); after an abort, only the own loads
      const int used = issued < STAGES ? (int)issued : STAGES;
      for (int i = 0; i < used; ++i) {
        // slot (stage - 1 - i) mod STAGES holds fill number issued - 1 - i
        const int s = (stage - 1 - i + 2 * STAGES) % STAGES;
        const uint32_t ph = (stage - 1 - i < 0) ? (phase ^ 1) : phase;
        if (ok) ok = mbar_wait(&empty[s], ph, abort, p.timeout_ns, p.status);
        if (!ok && (CG == 1 || leader)) mbar_wait_drain(&full[s], ph, p.timeout_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (the leader of a pair issues for both CTAs)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_make(1u /*bf16*/, TM, BN);
      // a single-CTA tile with at most 64 valid rows (a segment's tail) runs as M = 64: half
      // the MMA work; its rows land in the first 16 lanes of each TMEM lane quarter
      constexpr uint32_t idesc64 = idesc_make(1u, 64, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
        // tail tiles: A = the weight rows, B = the tokens (N = rows rounded up to 32)
        const uint32_t id = swap_tile(c.rows) ? idesc_make(1u, TM, (c.rows + 31) & ~31)
                                              : (CG == 1 && c.rows <= 64) ? idesc64 : idesc;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * S::kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * S::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {  // K = 16 per instruction: +32 bytes in the row
            if constexpr (CG == 1)
              mma_bf16(d_tmem, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + k * 32), id, (kb | k) != 0);
            else
              mma_bf16_pair(d_tmem, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + k * 32), id,
                            (kb | k) != 0);
          }
          // frees the stage (in both CTAs) once these MMAs have read it
          if constexpr (CG == 1) mma_commit(&empty[stage]);
          else mma_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if constexpr (CG == 1) mma_commit(&tfull[acc]);  // accumulator ready for the epilogue
        else mma_commit_pair(&tfull[acc], 0x3);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if constexpr (CG == 1) mma_commit(drain);  // completes when every MMA above has
      else mma_commit_pair(drain, 0x3);
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    } else if (lane == 0 && CG == 2) {
      // the pair's MMAs write this CTA's TMEM and read its shared memory: stay until done
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ======================= epilogue (warps 2..5; TMEM lane quarter = warp % 4)
    const int quarter = warp & 3;
    // 32 rows x 64 bytes per warp: bf16 rows leave through shared memory, coalesced
    uint8_t* stage = reinterpret_cast<uint8_t*>(seg_rows + kMaxGroups) + (warp - 2) * 2048;
    const uint32_t tempty_leader = CG == 2 ? mapa_shared(smem_addr(&tempty[0]), 0) : 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool dead = false;  // a wait gave up: the warp walks the rest of its tiles without work
    for (int tile = unit; tile < total_tiles; tile += nunits) {
      const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
      if (!dead) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort, p.timeout_ns, p.status));
        if (ok) tc_fence_after();
        else dead = true;
      }
      if (dead) {
        // every epilogue warp still meets each named barrier of the tail tiles' SwiGLU
        if (kSwiGLU && swap_tile(c.rows)) {
          for (int t0 = 0; t0 < c.rows; t0 += 32) {
            swap_bar();
            swap_bar();
          }
          swap_bar();
        }
        continue;
      }
      const bool extra = c.g >= p.G;
      if constexpr (kSwapTail) {
        if (swap_tile(c.rows)) {
          // TMEM lane = weight row, column = token. Token t is output row row0 + t.
          const int n = c.rows;
          const int64_t row0 = (extra ? p.out_extra_base : (int64_t)p.offsets[c.g]) + (int64_t)c.mb * TM;
          const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
          if (kSwiGLU) {
            // lanes 0-63 gate, 64-127 up of features f = 128 nb + 64 rank + fl; the up warps
            // hand their values to the gate warps through the four warps' staging areas, as
            // U[32 tokens][64 fl]. A barrier before each fill (no warp still uses its staging
            // for an earlier tile or chunk) and one after the tile (the next tile's stores).
            float* U = reinterpret_cast<float*>(seg_rows + kMaxGroups);
            const int fl = (quarter & 1) * 32 + lane;
            __nv_bfloat16* col = out + row0 * p.ldc + c.nb * (BN / 2) + (int)rank * 64 + fl;
            // EPI_SWIGLU_GU also keeps g and u: the tile's block of 128 g, then 128 u, of out2
            __nv_bfloat16* gcol = EPI == EPI_SWIGLU_GU ? static_cast<__nv_bfloat16*>(p.out2) + row0 * p.ldc2 +
                                                             c.nb * BN + (int)rank * 64 + fl
                                                       : nullptr;
            for (int t0 = 0; t0 < n; t0 += 32) {
              uint32_t v[32];
              tmem_ld32(t_row + t0, v);
              tmem_ld_wait();
              swap_bar();
              if (quarter >= 2) {
#pragma unroll
                for (int i = 0; i < 32; ++i) U[i * 64 + fl] = __uint_as_float(v[i]);
              }
              swap_bar();
              if (quarter < 2) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float g = __uint_as_float(v[i]), u = U[i * 64 + fl];
                  const float h = g / (1.0f + __expf(-g)) * u;
                  if (t0 + i < n) {
                    col[(int64_t)(t0 + i) * p.ldc] = __float2bfloat16_rn(h);
                    if (EPI == EPI_SWIGLU_GU) {
                      gcol[(int64_t)(t0 + i) * p.ldc2] = __float2bfloat16_rn(g);
                      gcol[(int64_t)(t0 + i) * p.ldc2 + BN / 2] = __float2bfloat16_rn(u);
                    }
                  }
                }
              }
            }
            swap_bar();
          } else {
            // lane = output feature 256 nb + 128 rank + 32 quarter + lane
            __nv_bfloat16* col = out + row0 * p.ldc + c.nb * BN + (int)rank * 128 + quarter * 32 + lane;
            for (int t0 = 0; t0 < n; t0 += 32) {
              uint32_t v[32];
              tmem_ld32(t_row + t0, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (t0 + i < n) col[(int64_t)(t0 + i) * p.ldc] = __float2bfloat16_rn(__uint_as_float(v[i]));
            }
          }
          tc_fence_before();
          __syncwarp();  // every lane's TMEM loads are complete: one arrival per warp
          if (lane == 0) {
            if (!leader) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
            else mbar_arrive_relaxed(&tempty[acc]);
          }
          if (++acc == 2) { acc = 0; acc_phase ^= 1; }
          continue;
        }
      }
      const bool m64 = CG == 1 && c.rows <= 64;  // M = 64 tile: 16 rows per lane quarter
      const int row_in_tile = m64 ? quarter * 16 + lane : (int)rank * BM + quarter * 32 + lane;
      const int64_t out_row = (extra ? p.out_extra_base : (int64_t)p.offsets[c.g]) + c.mb * TM + row_in_tile;
      const bool live = (!m64 || lane < 16) && row_in_tile < c.rows;
      // rows of this warp inside the segment (lane l holds warp row l; an M = 64 tile
      // gives a warp 16 rows)
      const int warp_live = min(c.rows - (row_in_tile - lane), m64 ? 16 : 32);
      const int64_t warp_row0 = out_row - lane;
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (EPI == EPI_SWIGLU_BF16 || EPI == EPI_SWIGLU_GU || EPI == EPI_SWIGLU_GATHER) {
        // cols [0, BN/2) gate, [BN/2, BN) up -> BN/2 columns of h
        uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + (warp_row0 * p.ldc + c.nb * (BN / 2)) * 2;
        uint8_t* out2 = EPI == EPI_SWIGLU_GU
                            ? reinterpret_cast<uint8_t*>(p.out2) + (warp_row0 * p.ldc2 + c.nb * BN) * 2
                            : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(t_row + c0, g);
          tmem_ld32(t_row + BN / 2 + c0, u);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float h0 = g0 / (1.0f + __expf(-g0)) * __uint_as_float(u[2 * i]);
            const float h1 = g1 / (1.0f + __expf(-g1)) * __uint_as_float(u[2 * i + 1]);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(h0, h1);
            packed[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
#pragma unroll
          for (int v = 0; v < 4; ++v)
            stage_piece(stage, lane, v, make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]));
          flush_rows_64B(stage, lane, out + 2 * c0, (int64_t)p.ldc * 2, warp_live);
          if (EPI == EPI_SWIGLU_GU) {
            // g and u as the backward reads them: the tile's block of 128 g, then 128 u
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t* src = half ? u : g;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 b2 =
                    __floats2bfloat162_rn(__uint_as_float(src[2 * i]), __uint_as_float(src[2 * i + 1]));
                packed[i] = *reinterpret_cast<const uint32_t*>(&b2);
              }
#pragma unroll
              for (int v = 0; v < 4; ++v)
                stage_piece(stage, lane, v,
                            make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]));
              flush_rows_64B(stage, lane, out2 + 2 * (c0 + half * (BN / 2)), (int64_t)p.ldc2 * 2, warp_live);
            }
          }
        }
      } else if (EPI == EPI_STORE_BF16 || EPI == EPI_STORE_GU) {
        uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + (warp_row0 * p.ldc + c.nb * BN) * 2;
        float rw = 1.0f;  // this lane's row weight (1 unless the routing weight is applied here)
        if (EPI == EPI_STORE_BF16 && p.w_topk != nullptr && !extra && live) {
          const int t = p.w_row_token[out_row];
          for (int j = 0; j < p.w_k; ++j)
            if (p.w_tok_row[(int64_t)t * p.w_k + j] == out_row) rw = p.w_topk[(int64_t)t * p.w_k + j];
        }
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(t_row + c0, v);
          tmem_ld_wait();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b2 =
                __floats2bfloat162_rn(rw * __uint_as_float(v[2 * i]), rw * __uint_as_float(v[2 * i + 1]));
            packed[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            stage_piece(stage, lane, q, make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]));
          flush_rows_64B(stage, lane, out + 2 * c0, (int64_t)p.ldc * 2, warp_live);
        }
      } else {
        float* out = reinterpret_cast<float*>(p.out) + out_row * p.ldc + c.nb * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(t_row + c0, v);
          tmem_ld_wait();
          if (live) {
            float4* dst = reinterpret_cast<float4*>(out + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 f = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
              if (p.bias) {
                const int n = c.nb * BN + c0 + 4 * q;
                f.x += p.bias[n]; f.y += p.bias[n + 1]; f.z += p.bias[n + 2]; f.w += p.bias[n + 3];
              }
              dst[q] = f;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();  // every lane's TMEM loads are complete: one arrival per warp
      if (lane == 0) {
        if (CG == 2 && !leader) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
        else mbar_arrive_relaxed(&tempty[acc]);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // neither CTA leaves while the pair still uses it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_cg<CG>(tmem_base, S::kTmemCols);
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major [rows, cols] matrix, box of box_rows x box_cols, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, cols] matrix copied box by box without swizzle (the shared-memory copy
// keeps the global byte order), e.g. the 512-byte MX scale atoms as rows of 128 uint32.
bool make_tmap_linear(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows,
                      uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool make_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, box_rows, BK);
}

}  // namespace

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

namespace {

template <int BN, int EPI, int CG = 1>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b0, const CUtensorMap& b1,
                   const CUtensorMap& b0x, const CUtensorMap& b1x, const TcParams& p, int64_t max_tiles,
                   cudaStream_t s, const SwapMaps* swp = nullptr) {
  if (max_tiles <= 0) return cudaSuccess;
  if (p.swap_rows > 0 && swp == nullptr) return cudaErrorInvalidValue;
  SwapMaps unused;  // no tail tiles: never read
  unused.t16 = unused.t16x = unused.g64 = unused.u64 = unused.g64x = unused.u64x = a;
  const SwapMaps& sw = swp ? *swp : unused;
  auto kern = tc_gemm_bf16_kernel<BN, EPI, CG>;
  const size_t smem = Smem<BN, CG>::kBytes;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if constexpr (CG == 1) {
    const int grid = (int)std::min<int64_t>(num_sms(), max_tiles);
    kern<<<grid, kThreads, smem, s>>>(a, a2, b0, b1, b0x, b1x, sw, p);
  } else {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a persistent grid must be resident all at once: no more pairs than fit together
    static int max_pairs = 0;
    if (!max_pairs) {
      cudaError_t e = cudaOccupancyMaxActiveClusters(&max_pairs, kern, &cfg);
      if (e != cudaSuccess || max_pairs <= 0) return e != cudaSuccess ? e : cudaErrorInvalidConfiguration;
    }
    const int pairs = (int)std::min<int64_t>(std::min(max_pairs, num_sms() / 2), max_tiles);
    cfg.gridDim = dim3(2 * pairs);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, a2, b0, b1, b0x, b1x, sw, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

bool router_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && (c.E == 128 || c.E == 256) && c.H % BK == 0;
}

bool mlp_supported(const moe_config_t& c) {
  if (encode_fn() == nullptr) return false;
  if (c.xfer_dtype == MOE_DTYPE_E4M3) return fp8_supported(c);
  if (c.xfer_dtype == MOE_DTYPE_MXE4M3) return mx_supported(c);
  if (c.act_dtype != MOE_DTYPE_BF16 || c.xfer_dtype != MOE_DTYPE_BF16) return false;
  return c.H % 128 == 0 && c.F % 128 == 0;
}

cudaError_t launch_router(const moe_config_t& c, const void* x, const void* w_router, const float* bias,
                          float* logits, DeviceStatus* st, cudaStream_t s) {
  // 128-wide N tiles (E / 128 tiles per 128 tokens) so that small T still spreads over the
  // SMs; with 256 experts and at least one 128-token tile per SM, one 256-wide N tile per
  // 128 tokens instead, which reads each token row once and halves the loads per flop
  const bool wide = c.E == 256 && ceil_div(c.T, BM) >= num_sms();
  const int bn = wide ? 256 : 128;
  CUtensorMap ta, tb;
  if (!make_bf16(&ta, x, c.T, c.H, BM) || !make_bf16(&tb, w_router, c.E, c.H, bn)) return cudaErrorInvalidValue;
  TcParams p{};
  p.G = 0;
  p.has_extra = 1;
  p.T_extra = c.T;
  p.a2_row_base = 0;
  p.out_extra_base = 0;
  p.K = c.H;
  p.n_tiles = c.E / bn;
  p.b_group_rows = 0;
  p.ldc = c.E;
  p.out = logits;
  p.bias = bias;
  p.timeout_ns = kTimeoutNs;
  p.status = st;
  const int64_t tiles = ceil_div(c.T, BM) * p.n_tiles;
  return wide ? launch<256, EPI_STORE_F32_BIAS>(ta, ta, tb, tb, tb, tb, p, tiles, s)
              : launch<128, EPI_STORE_F32_BIAS>(ta, ta, tb, tb, tb, tb, p, tiles, s);
}

cudaError_t launch_grouped_mlp(const moe_config_t& c, const void* xd, const float* xd_scale, const void* x,
                               const int32_t* offsets, const moe_weights_t& w, void* h, float* h_scale, void* yd,
                               DeviceStatus* st, cudaStream_t s, const int32_t* row_token, const int32_t* tok_row,
                               const float* topk_w, void* gu_keep) {
  if (c.xfer_dtype == MOE_DTYPE_E4M3)
    return launch_grouped_mlp_fp8(c, xd, xd_scale, offsets, w, h, h_scale, yd, st, s);
  // experts averaging fewer than 512 rows: the tokens go on the MMA's N axis, so an expert's
  // last tile is padded to a multiple of 32 tokens instead of 128 rows
  if (row_token == nullptr && topk_w == nullptr && gu_keep == nullptr && swap_supported(c) &&
      (int64_t)c.T * c.k < 512LL * c.E)
    return launch_grouped_mlp_swap(c, xd, x, offsets, w, h, yd, st, s);
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  // ---- GEMM1: h = silu(A Wg^T) * (A Wu^T), tiles of 128 h columns (256 B rows). A is the
  // dispatched rows xd, or (row_token given) the token rows of x gathered four at a time.
  CUtensorMap a1, a1x, bg, bu, bgx, bux;
  bool ok = (row_token ? make_bf16(&a1, x, c.T, c.H, 1) : make_bf16(&a1, xd, rows, c.H, BM)) &&
            make_bf16(&bg, w.w_gate, (uint64_t)c.E * c.F, c.H, 128) &&
            make_bf16(&bu, w.w_up, (uint64_t)c.E * c.F, c.H, 128);
  if (shared) {
    ok = ok && make_bf16(&a1x, x, c.T, c.H, BM) && make_bf16(&bgx, w.ws_gate, c.F, c.H, 128) &&
         make_bf16(&bux, w.ws_up, c.F, c.H, 128);
  } else {
    a1x = a1; bgx = bg; bux = bu;
  }
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = 0;
  p.out_extra_base = R;
  p.K = c.H;
  p.n_tiles = c.F / 128;
  p.b_group_rows = c.F;
  p.ldc = c.F;
  p.out = h;
  p.row_token = row_token;
  p.a_rows = static_cast<const uint8_t*>(x);
  p.a_ld_bytes = (int64_t)c.H * 2;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  // CTA pairs (256-row tiles) when experts average at least 512 rows; with fewer rows the
  // second 128 rows of a pair tile would mostly be padding.
  const bool pair = (int64_t)c.T * c.k >= 512LL * c.E && c.H % 256 == 0;
  const int tm = pair ? 2 * BM : BM;
  const int64_t mt_bound = ceil_div(R, tm) + c.E + (shared ? ceil_div(c.T, tm) : 0);
  cudaError_t e;
  // The keep epilogue reads A by TMA boxes: gathered rows reach it only as CTA pairs, whose
  // producers gather with TMA; single CTAs gather with cp.async in their own epilogue mode.
  if (gu_keep != nullptr && row_token != nullptr && !pair) return cudaErrorInvalidValue;
  // CTA pairs without row gathers: segment tails of at most kSwapRows rows run with their
  // tokens on the MMA's N axis
  SwapMaps sw;
  const bool tails = pair && row_token == nullptr;
  if (tails) {
    ok = make_bf16(&sw.t16, xd, rows, c.H, 16) && make_bf16(&sw.g64, w.w_gate, (uint64_t)c.E * c.F, c.H, 64) &&
         make_bf16(&sw.u64, w.w_up, (uint64_t)c.E * c.F, c.H, 64);
    if (shared) {
      ok = ok && make_bf16(&sw.t16x, x, c.T, c.H, 16) && make_bf16(&sw.g64x, w.ws_gate, c.F, c.H, 64) &&
           make_bf16(&sw.u64x, w.ws_up, c.F, c.H, 64);
    } else {
      sw.t16x = sw.t16; sw.g64x = sw.g64; sw.u64x = sw.u64;
    }
    if (!ok) return cudaErrorInvalidValue;
  }
  if (gu_keep != nullptr) {  // also keep g and u for the backward
    p.out2 = gu_keep;
    p.ldc2 = 2 * c.F;
    p.swap_rows = tails ? kSwapRows : 0;
    e = pair ? launch<256, EPI_SWIGLU_GU, 2>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s, tails ? &sw : nullptr)
             : launch<256, EPI_SWIGLU_GU, 1>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
    p.out2 = nullptr;
    p.swap_rows = 0;
  } else {
    if (tails) {
      p.swap_rows = kSwapRows;
      e = launch<256, EPI_SWIGLU_BF16, 2>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s, &sw);
      p.swap_rows = 0;
    } else if (pair)
      e = launch<256, EPI_SWIGLU_BF16, 2>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
    else if (row_token)  // single CTAs gather their rows with cp.async
      e = launch<256, EPI_SWIGLU_GATHER, 1>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
    else
      e = launch<256, EPI_SWIGLU_BF16, 1>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
  }
  if (e != cudaSuccess) return e;
  // ---- GEMM2: yd = h Wd^T (the shared expert's h rows follow the routed ones)
  const int bn2 = c.H % 256 == 0 ? 256 : 128;
  const uint32_t box2 = pair ? bn2 / 2 : bn2;  // a pair's CTAs each load half of the N tile
  CUtensorMap a2, bd, bdx;
  ok = make_bf16(&a2, h, rows, c.F, BM) && make_bf16(&bd, w.w_down, (uint64_t)c.E * c.H, c.F, box2);
  if (shared) ok = ok && make_bf16(&bdx, w.ws_down, c.H, c.F, box2);
  else bdx = bd;
  if (!ok) return cudaErrorInvalidValue;
  p.a2_row_base = (int)R;
  p.row_token = nullptr;
  if (topk_w != nullptr) {  // routing weights in GEMM2's epilogue (row_token and tok_row given)
    p.w_row_token = row_token;
    p.w_tok_row = tok_row;
    p.w_topk = topk_w;
    p.w_k = c.k;
  }
  p.K = c.F;
  p.n_tiles = c.H / bn2;
  p.b_group_rows = c.H;
  p.ldc = c.H;
  p.out = yd;
  if (pair && topk_w == nullptr) {
    // segment tails of at most kSwapRows rows run with their tokens on the MMA's N axis (the
    // routed and the shared expert's h rows come from the same map)
    SwapMaps sw2;
    if (!make_bf16(&sw2.t16, h, rows, c.F, 16)) return cudaErrorInvalidValue;
    sw2.t16x = sw2.t16;
    sw2.g64 = sw2.u64 = sw2.g64x = sw2.u64x = bd;  // GEMM2's tail tiles load their weights through bd / bdx
    p.swap_rows = kSwapRows;
    return launch<256, EPI_STORE_BF16, 2>(a2, a2, bd, bd, bdx, bdx, p, mt_bound * p.n_tiles, s, &sw2);
  }
  if (pair) return launch<256, EPI_STORE_BF16, 2>(a2, a2, bd, bd, bdx, bdx, p, mt_bound * p.n_tiles, s);
  if (bn2 == 256) return launch<256, EPI_STORE_BF16, 1>(a2, a2, bd, bd, bdx, bdx, p, mt_bound * p.n_tiles, s);
  return launch<128, EPI_STORE_BF16, 1>(a2, a2, bd, bd, bdx, bdx, p, mt_bound * p.n_tiles, s);
}

cudaError_t launch_gate_up_preact(const moe_config_t& c, const void* xd, const void* x, const int32_t* offsets,
                                  const moe_weights_t& w, void* gu, DeviceStatus* st, cudaStream_t s) {
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  // the operands, tiles and CTA-pair choice of the forward's GEMM1 (the shared expert's A = x)
  CUtensorMap a1, a1x, bg, bu, bgx, bux;
  bool ok = make_bf16(&a1, xd, rows, c.H, BM) && make_bf16(&bg, w.w_gate, (uint64_t)c.E * c.F, c.H, 128) &&
            make_bf16(&bu, w.w_up, (uint64_t)c.E * c.F, c.H, 128);
  if (shared) {
    ok = ok && make_bf16(&a1x, x, c.T, c.H, BM) && make_bf16(&bgx, w.ws_gate, c.F, c.H, 128) &&
         make_bf16(&bux, w.ws_up, c.F, c.H, 128);
  } else {
    a1x = a1; bgx = bg; bux = bu;
  }
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = 0;
  p.out_extra_base = R;
  p.K = c.H;
  p.n_tiles = c.F / 128;
  p.b_group_rows = c.F;
  p.ldc = 2 * c.F;
  p.out = gu;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  const bool pair = (int64_t)c.T * c.k >= 512LL * c.E && c.H % 256 == 0;
  const int tm = pair ? 2 * BM : BM;
  const int64_t mt_bound = ceil_div(R, tm) + c.E + (shared ? ceil_div(c.T, tm) : 0);
  return pair ? launch<256, EPI_STORE_GU, 2>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s)
              : launch<256, EPI_STORE_GU, 1>(a1, a1x, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
}

}  // namespace tc
}  // namespace moe
