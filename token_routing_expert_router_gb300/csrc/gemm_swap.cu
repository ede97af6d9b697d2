// Grouped expert GEMMs for experts with few rows each: the tokens on the MMA's N axis.
//
// With ~256 rows an expert (the DeepSeek-V3 shape: 256 experts, top-8), 128-row tiles over
// each expert's rows leave the last tile of most experts partly empty. The grouped GEMM
// ("Scalable Training of Mixture-of-Experts Models with Megatron Core" summary, section
// 2.4: all experts' GEMMs in one kernel, shapes read on the device) is written here as
// D^T = W . A^T: the MMA's M side is 256 weight rows, split over a CTA pair
// (tcgen05.mma.cta_group::2, each CTA 128 rows of its own), and its N side is the expert's
// tokens in multiples of 32 (each CTA loads half of them).
//
// A tile takes up to 512 of a group's tokens against one 256-row weight block: tokens
// [0, 256) accumulate in one 256-column TMEM slot and tokens [256, 512) in the other, both
// MMAs reading the same weight stage. On this shape the operands' trip from L2 into the SMs
// is what limits the GEMM, and a weight block read once for up to 512 tokens halves the
// weight share of that traffic for experts with more than 256 rows. Tiles of at most 256
// tokens take one slot, alternating, so their epilogue overlaps the next tile's MMAs.
//
// TMEM then holds features on lanes and tokens on columns; the epilogue transposes through
// shared memory so that every store writes rows of the output.
//   GEMM1 (gate/up + SwiGLU): CTA r holds the gate rows and the up rows of 64 features
//     (64 + 64 = 128 TMEM lanes). Lane quarters 0/1 hold g, quarters 2/3 hold u for the
//     same features; the two warps of a feature range trade half of their tokens through
//     shared memory, each computes h = silu(g) * u for 16 of every 32 tokens.
//   GEMM2 (down): CTA r holds 128 output features.
// Block: warp 0 TMA producer, warp 1 MMA issuer (the leader CTA issues for the pair),
// warps 2-9 epilogue (two per TMEM lane quarter, taking alternate 32-token chunks).
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "tc_common.cuh"

namespace moe {
namespace tc {

bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols);
int num_sms();

namespace {

constexpr int BK = 64;                           // bf16 K per stage: one 128-byte swizzle row
constexpr int kWRows = 128;                      // weight rows per CTA (the pair's M = 256)
constexpr int kSlotTok = 256;                    // tokens per TMEM slot (the MMA's N at most)
constexpr int kMaxTok = 2 * kSlotTok;            // tokens per tile
constexpr int kTokAlign = 32;                    // N granularity (each CTA: multiples of 16 rows)
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxGroups = 514;
constexpr uint64_t kTimeoutNs = 2000000000ull;   // 2 s: no legitimate wait comes close
constexpr int kABytes = kWRows * BK * 2;         // 16 KB of weight rows
constexpr int kBHalf = (kSlotTok / 2) * BK * 2;  // 16 KB: one slot's token rows of this CTA
constexpr int kBBytes = 2 * kBHalf;
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kStages = 4;
constexpr int kSlotCols = 256;
constexpr int kTmemCols = 2 * kSlotCols;
constexpr int kStagingBytes = kEpiWarps * 2048;  // 32 rows x 64 B per epilogue warp
constexpr size_t kSmemBytes =
    1024 + (size_t)kStages * kStageBytes + 256 + 2 * kMaxGroups * sizeof(int32_t) + kStagingBytes;

enum { SW_SWIGLU = 0, SW_STORE = 1 };

struct SwMaps {
  CUtensorMap w0, w1;    // routed weights: GEMM1 gate and up [E*F, H] (64-row boxes); GEMM2 down [E*H, F] (128)
  CUtensorMap w0x, w1x;  // the extra group's (shared expert's) weights
  CUtensorMap t[4];      // routed token rows (GEMM1: xd; GEMM2: h), boxes of 128, 64, 32, 16 rows
  CUtensorMap tx[4];     // the extra group's token rows (GEMM1: x; GEMM2: h)
};

struct SwParams {
  const int32_t* offsets;  // [G+1] routed segment starts (device)
  int G;                   // routed groups
  int has_extra;           // one more group of T_extra tokens (the shared expert)
  int T_extra;
  int a2_row_base;         // row of the extra group's token 0 in tx
  int64_t out_extra_base;  // output row of the extra group's token 0
  int K;                   // reduction length, multiple of BK
  int n_fb;                // feature blocks per group (GEMM1: F / 128; GEMM2: H / 256)
  int w_group_rows;        // weight rows per routed group (GEMM1: F; GEMM2: H)
  int ldc;                 // output row length in elements
  void* out;
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// Tokens [begin, begin + len) of a group's token tile mb (512 tokens a tile): n0 MMA
// columns for tokens [begin, begin + 256) in the first slot and, for len > 256, n1 columns
// for the rest in the second (both multiples of 32; n1 = 0: one slot).
struct TokTile {
  int begin, len, n0, n1;
};

__device__ __forceinline__ int round_tok(int n) { return (n + kTokAlign - 1) / kTokAlign * kTokAlign; }

__device__ __forceinline__ TokTile tok_tile(int rows, int mb) {
  TokTile t;
  t.begin = mb * kMaxTok;
  t.len = min(kMaxTok, rows - t.begin);
  t.n0 = t.len > kSlotTok ? kSlotTok : round_tok(t.len);
  t.n1 = t.len > kSlotTok ? round_tok(t.len - kSlotTok) : 0;
  return t;
}

// The TMEM slots a tile uses: a two-part tile takes slots 0 and 1; a one-part tile takes
// the slot after the previous one-part tile's (slot 0 after a two-part tile), so that
// consecutive one-part tiles alternate. The MMA issuer and the epilogue both walk it.
struct SlotWalk {
  int cur = 0;
  uint32_t uses0 = 0, uses1 = 0;  // uses of each slot before the current tile
  __device__ __forceinline__ int first(bool two) const { return two ? 0 : cur; }
  __device__ __forceinline__ uint32_t uses(int slot) const { return slot ? uses1 : uses0; }
  __device__ __forceinline__ void advance(bool two) {
    if (two || cur == 0) ++uses0;
    if (two || cur == 1) ++uses1;
    cur = two ? 0 : cur ^ 1;
  }
};

// One bf16 of staging row j (a token), column `lane` (a feature), in the swizzled layout
// flush_rows_64B reads: piece c of row j at j * 64 + 16 * (c ^ ((j >> 1) & 3)). For a fixed j
// the 32 lanes write the row's 64 contiguous bytes (no bank conflict).
__device__ __forceinline__ void stage_bf16(uint8_t* stage, int j, int lane, float v) {
  *reinterpret_cast<__nv_bfloat16*>(stage + j * 64 + 16 * ((lane >> 3) ^ ((j >> 1) & 3)) + 2 * (lane & 7)) =
      __float2bfloat16_rn(v);
}

// The first 16 staged rows to global memory (8 rows x 64 bytes per store instruction).
__device__ __forceinline__ void flush_rows_64B_16(uint8_t* stage, int lane, uint8_t* base, int64_t stride, int live) {
  __syncwarp();
  const int c = lane & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int row = 8 * j + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4*>(stage + row * 64 + 16 * (c ^ ((row >> 1) & 3)));
    if (row < live) *reinterpret_cast<uint4*>(base + row * stride + 16 * c) = v;
  }
  __syncwarp();
}

__device__ __forceinline__ void pair_bar_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// `rows` token rows (a multiple of 16, at most 128) as boxes of 128, or of 64, 32 and 16
// rows (the bits of rows / 16), into consecutive rows of dst.
__device__ __forceinline__ void load_tokens(const CUtensorMap* tmaps, uint8_t* dst, uint32_t bar, int x, int row,
                                            int rows) {
  if (rows == 128) {
    tma_load_2d_pair(&tmaps[0], dst, bar, x, row);
    return;
  }
  int off = 0;
#pragma unroll
  for (int bi = 1; bi < 4; ++bi) {
    const int box = 128 >> bi;
    if (rows & box) {
      tma_load_2d_pair(&tmaps[bi], dst + off * BK * 2, bar, x, row + off);
      off += box;
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) tc_swap_kernel(const __grid_constant__ SwMaps maps, const SwParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;  // [2] per TMEM slot
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(bars + 32);  // [ngroups + 1]
  int32_t* seg_rows = mt_prefix + kMaxGroups;                 // [ngroups]
  uint8_t* staging = reinterpret_cast<uint8_t*>(seg_rows + kMaxGroups);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.G + p.has_extra;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int unit = blockIdx.x / 2, nunits = gridDim.x / 2;  // tile walkers: CTA pairs

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * 32 * kEpiWarps);  // every epilogue thread of both CTAs
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&maps.w0);
    if (EPI == SW_SWIGLU) tma_prefetch_desc(&maps.w1);
    tma_prefetch_desc(&maps.t[0]);
  }
  if (warp == 1) tmem_alloc_cg<2>(tmem_slot, kTmemCols);
  if (warp == 2) build_tile_prefix(p.offsets, p.G, ngroups, p.T_extra, kMaxTok, lane, seg_rows, mt_prefix);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.n_fb * mt_prefix[ngroups];
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ======================= TMA producer: every CTA loads its own weight rows and its
    // half of each slot's tokens; both CTAs' loads complete on the leader's barrier
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_fb, seg_rows, kMaxTok);
        const bool extra = c.g >= p.G;
        const TokTile tt = tok_tile(seg_rows[c.g], c.mb);
        const int h0 = tt.n0 / 2, h1 = tt.n1 / 2;  // this CTA's token rows of each slot
        const int tbase = (extra ? p.a2_row_base : p.offsets[c.g]) + tt.begin;
        const int trow0 = tbase + (int)rank * h0, trow1 = tbase + kSlotTok + (int)rank * h1;
        const CUtensorMap* tmaps = extra ? maps.tx : maps.t;
        const CUtensorMap* w0 = extra ? &maps.w0x : &maps.w0;
        const CUtensorMap* w1 = extra ? &maps.w1x : &maps.w1;
        const int wg = extra ? 0 : c.g * p.w_group_rows;
        // GEMM1: gate and up rows of features [128 nb + 64 r, +64); GEMM2: rows [256 nb + 128 r, +128)
        const int wrow = EPI == SW_SWIGLU ? wg + c.nb * 128 + (int)rank * 64 : wg + c.nb * 256 + (int)rank * 128;
        const uint32_t bytes = 2u * (uint32_t)(kABytes + (h0 + h1) * BK * 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * kBBytes;
          if (leader) mbar_arrive_expect_tx(&full[stage], bytes);
          const uint32_t bar = mapa_shared(smem_addr(&full[stage]), 0);
          if (EPI == SW_SWIGLU) {
            tma_load_2d_pair(w0, a_dst, bar, kb * BK, wrow);                 // 64 gate rows
            tma_load_2d_pair(w1, a_dst + 64 * BK * 2, bar, kb * BK, wrow);  // 64 up rows
          } else {
            tma_load_2d_pair(w0, a_dst, bar, kb * BK, wrow);
          }
          load_tokens(tmaps, b_dst, bar, kb * BK, trow0, h0);
          if (h1) load_tokens(tmaps, b_dst + kBHalf, bar, kb * BK, trow1, h1);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // tail: every stage's last fill has been consumed, so no TMA write or MMA read is still
      // in flight when the block exits; after an abort, the leader drains its own barriers
      const int used = issued < kStages ? (int)issued : kStages;
      for (int i = 0; i < used; ++i) {
        const int s = (stage - 1 - i + 2 * kStages) % kStages;
        const uint32_t ph = (stage - 1 - i < 0) ? (phase ^ 1) : phase;
        if (ok) ok = mbar_wait(&empty[s], ph, abort, p.timeout_ns, p.status);
        if (!ok && leader) mbar_wait_drain(&full[s], ph, p.timeout_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer: the leader issues M = 256 pair MMAs, N = a slot's tokens
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      SlotWalk sw;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_fb, seg_rows, kMaxTok);
        const TokTile tt = tok_tile(seg_rows[c.g], c.mb);
        const bool two = tt.n1 > 0;
        const int s0 = sw.first(two);
        const uint32_t id0 = idesc_make(1u /*bf16*/, 256, tt.n0);
        const uint32_t id1 = idesc_make(1u, 256, two ? tt.n1 : 32);
        if (!mbar_wait(&tempty[s0], (sw.uses(s0) & 1) ^ 1, abort, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + s0 * kSlotCols, d1 = tmem_base + kSlotCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)  // K = 16 per instruction: +32 bytes in the row
            mma_bf16_pair(d0, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + k * 32), id0, (kb | k) != 0);
          if (two) {
            // the second slot is waited for only now, so the first slot's MMAs of this K
            // block already run while its previous tile's epilogue finishes
            if (kb == 0) {
              if (!mbar_wait(&tempty[1], (sw.uses(1) & 1) ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
              tc_fence_after();
            }
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              mma_bf16_pair(d1, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + kBHalf + k * 32), id1,
                            (kb | k) != 0);
          }
          mma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs once read
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit_pair(&tfull[s0], 0x3);  // slots ready for both CTAs' epilogues
        if (two) mma_commit_pair(&tfull[1], 0x3);
        sw.advance(two);
      }
      mma_commit_pair(drain, 0x3);  // completes when every MMA above has
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    } else if (lane == 0) {
      // the pair's MMAs write this CTA's TMEM and read its shared memory: stay until done
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ======================= epilogue (warps 2..9; TMEM lane quarter = warp % 4; the two
    // warps of a quarter take alternate 32-token chunks)
    const int quarter = warp & 3;
    const int local = (warp - 2) & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = staging + (warp - 2) * 2048;
    // GEMM1: quarters 0/1 hold g and quarters 2/3 u of the same 32 features (range quarter & 1);
    // the partner warp has the same half and the other quarter of the range
    const bool is_gate = quarter < 2;
    const int range = quarter & 1;
    const uint8_t* partner_stg = staging + (4 * half + (local ^ 2)) * 2048;
    const int bar_id = 1 + range + 2 * half;
    const uint32_t tempty_leader = mapa_shared(smem_addr(&tempty[0]), 0);
    SlotWalk sw;
    bool ok = true;
    for (int tile = unit; tile < total_tiles; tile += nunits) {
      const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_fb, seg_rows, kMaxTok);
      const bool extra = c.g >= p.G;
      const TokTile tt = tok_tile(seg_rows[c.g], c.mb);
      const bool two = tt.n1 > 0;
      const int64_t row0 = (extra ? p.out_extra_base : (int64_t)p.offsets[c.g]) + tt.begin;  // token 0's row
      for (int part = 0; part < (two ? 2 : 1); ++part) {
        const int slot = part == 0 ? sw.first(two) : 1;
        const int n = part == 0 ? tt.n0 : tt.n1;
        const int tok_base = part * kSlotTok;  // first token of this slot, within the tile
        // After an abort the GEMM1 warps keep walking the tiles' chunks without waiting or
        // loading, so that both warps of a pair reach every barrier they share.
        if (ok) ok = mbar_wait(&tfull[slot], sw.uses(slot) & 1, abort, p.timeout_ns, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok && EPI == SW_STORE) break;
        if (ok) tc_fence_after();
        const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + slot * kSlotCols;
        bool released = false;
        auto release = [&]() {  // this warp's last TMEM read of the slot is complete
          if (ok && !released) {
            tc_fence_before();
            if (!leader) mbar_arrive_cluster_relaxed(tempty_leader + slot * 8);
            else mbar_arrive_relaxed(&tempty[slot]);
          }
          released = true;
        };
        if (EPI == SW_STORE) {
          const int feat0 = c.nb * 256 + (int)rank * 128 + quarter * 32;  // this warp's 32 output features
          uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + ((row0 + tok_base) * p.ldc + feat0) * 2;
#pragma unroll 1
          for (int c0 = 32 * half; c0 < n; c0 += 64) {
            uint32_t v[32];
            tmem_ld32(t_row + c0, v);
            tmem_ld_wait();
            if (c0 + 64 >= n) release();
#pragma unroll
            for (int j = 0; j < 32; ++j) stage_bf16(stg, j, lane, __uint_as_float(v[j]));
            flush_rows_64B(stg, lane, out + (int64_t)c0 * p.ldc * 2, (int64_t)p.ldc * 2,
                           tt.len - tok_base - c0);
          }
        } else {
          const int feat0 = c.nb * 128 + (int)rank * 64 + range * 32;  // this range's 32 h columns
          uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + ((row0 + tok_base) * p.ldc + feat0) * 2;
#pragma unroll 1
          for (int c0 = 32 * half; c0 < n; c0 += 64) {
            uint32_t v[32];
            if (ok) {
              tmem_ld32(t_row + c0, v);
              tmem_ld_wait();
              if (c0 + 64 >= n) release();
              // the gate warp sends g of tokens 16..31 and keeps 0..15; the up warp sends u of
              // tokens 0..15 and keeps 16..31, each through its own staging buffer ([token][lane])
              float* send = reinterpret_cast<float*>(stg);
#pragma unroll
              for (int i = 0; i < 16; ++i) send[i * 32 + lane] = __uint_as_float(v[is_gate ? 16 + i : i]);
            }
            pair_bar_sync(bar_id);
            float r[16];
            if (ok) {
              const float* recv = reinterpret_cast<const float*>(partner_stg);
#pragma unroll
              for (int i = 0; i < 16; ++i) r[i] = recv[i * 32 + lane];
            }
            pair_bar_sync(bar_id);  // the partner has read this warp's buffer: reuse it
            if (ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float g = is_gate ? __uint_as_float(v[i]) : r[i];
                const float u = is_gate ? r[i] : __uint_as_float(v[16 + i]);
                stage_bf16(stg, i, lane, g / (1.0f + __expf(-g)) * u);
              }
              const int tok0 = c0 + (is_gate ? 0 : 16);
              flush_rows_64B_16(stg, lane, out + (int64_t)tok0 * p.ldc * 2, (int64_t)p.ldc * 2,
                                tt.len - tok_base - tok0);
            }
          }
        }
        release();  // a warp without chunks in this slot hands it back at once
      }
      if (!ok && EPI == SW_STORE) break;
      sw.advance(two);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair still uses it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_cg<2>(tmem_base, kTmemCols);
  }
}

bool make_bf16_box(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, box_rows, BK);
}

// The four token-row maps of one tensor (boxes of 128, 64, 32 and 16 rows).
bool make_token_maps(CUtensorMap (&m)[4], const void* base, uint64_t rows, uint64_t cols) {
  for (int i = 0; i < 4; ++i)
    if (!make_bf16_box(&m[i], base, rows, cols, 128u >> i)) return false;
  return true;
}

template <int EPI>
cudaError_t launch_swap(const SwMaps& maps, const SwParams& p, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  auto kern = tc_swap_kernel<EPI>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * (num_sms() / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool swap_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.xfer_dtype == MOE_DTYPE_BF16 && c.H % 256 == 0 && c.F % 128 == 0 &&
         c.E <= kMaxGroups - 2;
}

cudaError_t launch_grouped_mlp_swap(const moe_config_t& c, const void* xd, const void* x, const int32_t* offsets,
                                    const moe_weights_t& w, void* h, void* yd, DeviceStatus* st, cudaStream_t s) {
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  // ---- GEMM1: h = silu(A Wg^T) * (A Wu^T); routed A = xd, the shared expert's A = x
  SwMaps m1{};
  bool ok = make_bf16_box(&m1.w0, w.w_gate, (uint64_t)c.E * c.F, c.H, 64) &&
            make_bf16_box(&m1.w1, w.w_up, (uint64_t)c.E * c.F, c.H, 64) && make_token_maps(m1.t, xd, R, c.H);
  if (shared) {
    ok = ok && make_bf16_box(&m1.w0x, w.ws_gate, c.F, c.H, 64) && make_bf16_box(&m1.w1x, w.ws_up, c.F, c.H, 64) &&
         make_token_maps(m1.tx, x, c.T, c.H);
  } else {
    m1.w0x = m1.w0;
    m1.w1x = m1.w1;
    for (int i = 0; i < 4; ++i) m1.tx[i] = m1.t[i];
  }
  if (!ok) return cudaErrorInvalidValue;
  SwParams p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = 0;
  p.out_extra_base = R;
  p.K = c.H;
  p.n_fb = c.F / 128;
  p.w_group_rows = c.F;
  p.ldc = c.F;
  p.out = h;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  // token tiles: at most ceil(rows / 512) per group
  const int64_t tt_bound = ceil_div(R, kMaxTok) + c.E + (shared ? ceil_div(c.T, kMaxTok) : 0);
  cudaError_t e = launch_swap<SW_SWIGLU>(m1, p, tt_bound * p.n_fb, s);
  if (e != cudaSuccess) return e;
  // ---- GEMM2: yd = h Wd^T (the shared expert's h rows follow the routed ones)
  SwMaps m2{};
  ok = make_bf16_box(&m2.w0, w.w_down, (uint64_t)c.E * c.H, c.F, 128) && make_token_maps(m2.t, h, rows, c.F);
  if (shared) ok = ok && make_bf16_box(&m2.w0x, w.ws_down, c.H, c.F, 128);
  else m2.w0x = m2.w0;
  if (!ok) return cudaErrorInvalidValue;
  m2.w1 = m2.w0;
  m2.w1x = m2.w0x;
  for (int i = 0; i < 4; ++i) m2.tx[i] = m2.t[i];
  p.a2_row_base = (int)R;
  p.K = c.F;
  p.n_fb = c.H / 256;
  p.w_group_rows = c.H;
  p.ldc = c.H;
  p.out = yd;
  return launch_swap<SW_STORE>(m2, p, tt_bound * p.n_fb, s);
}

}  // namespace tc
}  // namespace moe
