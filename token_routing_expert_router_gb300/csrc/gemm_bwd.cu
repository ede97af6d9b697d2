// Backward of the grouped expert MLP (bf16 layers) on the tcgen05 tensor cores.
//
// The backward of the experts' grouped GEMM ("Scalable Training of Mixture-of-Experts
// Models with Megatron Core" summary, section 2.4 grouped GEMM, which serves the training
// step in both directions; section 2.2 recomputation instead of stored activations) is
// four grouped GEMMs over the same expert segments as the forward:
//   DGRAD_DOWN  dh  = dyd . Wd            K = H, B = Wd read MN-major (its rows are the K
//               index), fused epilogue: g and u (recomputed by the forward GEMM1 kernel
//               into gu) give h = silu(g) u and the SwiGLU backward dg, du -> dgu, h
//   DGRAD_GU    dxd = dg . Wg + du . Wu   K = 2F (dgu's interleaved gate/up blocks), B =
//               Wg or Wu per K block, read MN-major
//   WGRAD_DOWN  dWd[e] = dyd_e^T . h_e    K = the expert's token rows, both operands
//               MN-major (an activation's rows are the K index)
//   WGRAD_GU    dWg[e], dWu[e] = dgu_e^T . xd_e
//   DGRAD_PLAIN C = A . B                 K-major A, B read MN-major (its rows are the K
//               index), a plain bf16 store: the router's share of the input gradient,
//               dl . W_router, over the tokens as one group (the router's weight gradient
//               dl^T . x is WGRAD_DOWN over that group)
// An MN-major operand is loaded by TMA as boxes of 64 MN elements (128 bytes, 128-byte
// swizzle) x 64 K rows; its shared-memory descriptor has LBO = the byte distance between
// the 64-element MN blocks (8 KB here), SBO = 1024 B between 8-row K groups, and each MMA
// of K = 16 advances the start by 16 rows (2 KB). Instruction-descriptor bits 15 / 16 mark
// A / B as MN-major.
// Wgrad reduces over an expert's rows in K stages of 64, and the last stage of a segment
// reaches past its end. dgu and h, which the backward writes itself, are therefore laid out
// with every expert's rows padded to a multiple of 64 by zero rows: expert g (the shared
// expert is g = E at offset T*k) starts at padded row P(g) = 64 * ceil((offsets[g] + 63 g) /
// 64), which needs no prefix sum and never overlaps the next expert. Each wgrad pairs one
// padded operand (dgu, or h) with an unpadded one (xd, or dyd): past the segment's end the
// padded operand's rows are zero, so the other's rows (the next expert's, or the TMA's
// zero fill past the end of the map) add nothing. An expert without rows gets an all-zero
// gradient from the epilogue without touching the tensor core.
//
// Block: warp 0 TMA producer, warp 1 MMA issuer (TMEM owner), warps 2-9 epilogue (one
// output row per thread, two warps per TMEM lane quarter each owning 128 of the tile's 256
// columns; two TMEM accumulators of 256 columns). Weight-gradient tiles are short (K = one
// expert's rows) and write 128 KB of fp32 per CTA each, so the epilogue must keep pace with
// a few microseconds of MMAs: eight warps, and TMEM loads issued one chunk ahead.
// Tiles of 128 x 256 (one CTA) or 256 x 256 (a CTA pair, M = 256 pair MMAs, each CTA
// holding half of B: 6 stages of 32 KB instead of 4 of 48 KB), K stages of 64 (128 bytes).
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "tc_common.cuh"

namespace moe {
namespace tc {

bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols);
int num_sms();

namespace {

constexpr int BM = 128, BN = 256, BK = 64;  // BK in bf16 elements (128 bytes)
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kABytes = BM * BK * 2;  // 16 KB: this CTA's 128 rows of A
constexpr int kMaxGroups = 514;
constexpr int kTmemCols = 2 * BN;
constexpr uint64_t kTimeoutNs = 2000000000ull;

// Shared memory of one CTA. A CTA pair (CG = 2) holds half of B's 256 columns per CTA, so a
// stage is 32 KB and six stages fit instead of four.
template <int CG>
struct BwdSmem {
  static constexpr int kBBytes = (BN / CG) * BK * 2;  // (BN / CG) / 64 MN boxes of 8 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = CG == 2 ? 6 : 4;
  static constexpr size_t kBytes =
      1024 + (size_t)kStages * kStageBytes + 256 + 2 * kMaxGroups * sizeof(int32_t) + kEpiWarps * 2048;
};

enum Mode { DGRAD_DOWN = 0, DGRAD_GU = 1, WGRAD_DOWN = 2, WGRAD_GU = 3, DGRAD_PLAIN = 4 };

struct BwdParams {
  const int32_t* offsets;
  int G, has_extra, T_extra, a2_row_base;  // the shared expert's rows: [a2_row_base, + T_extra)
  int K;             // dgrad: the contraction length (H or 2F)
  int n_tiles;       // 256-wide N tiles (dgrad: N/256; wgrad: N_out/256)
  int m_tiles_out;   // wgrad: M_out / (128 * CG)
  int b_group_rows;  // dgrad: rows of B per routed group in its map (H for Wd, F for Wg/Wu)
  int F;
  int ldc;                    // dgrad output row length (elements)
  __nv_bfloat16* out;         // DGRAD_DOWN: dgu [prows, 2F]; DGRAD_GU: dxd [rows, H]
  __nv_bfloat16* h_out;       // DGRAD_DOWN: h [prows, F]
  const __nv_bfloat16* gu;    // DGRAD_DOWN: g and u [rows, 2F], interleaved in 128-column blocks
  float* w0;                  // WGRAD_DOWN: dWd [G, M_out, N_out]; WGRAD_GU: dWg [G, F, H]
  float* w1;                  // WGRAD_GU: dWu [G, F, H]
  float* w0x;                 // the shared expert's (same layouts without the G dimension)
  float* w1x;
  int M_out, N_out;
  int extra_b_row0;           // WGRAD_GU: the shared expert's first row in its B map (x)
  int b_unpadded;             // WGRAD_DOWN: B's rows are the groups' own rows (not padded h);
                              //   every group but the last then spans whole 64-row K stages
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// First padded row of group g (offset = its first row in the unpadded buffers).
__host__ __device__ __forceinline__ int64_t padded_row0(int64_t offset, int g) {
  return (offset + 63 * (int64_t)g + 63) / 64 * 64;
}

// Weight-gradient tiles: per group, m_tiles x n_tiles output tiles (mb, nb) of the gradient;
// rows = the group's token rows, the tile's reduction length.
__device__ __forceinline__ TileCoord decode_wgrad(int tile, int m_tiles, int n_tiles, const int32_t* seg_rows) {
  const int per = m_tiles * n_tiles;
  TileCoord c;
  c.g = tile / per;
  const int local = tile - c.g * per;
  c.mb = local / n_tiles;
  c.nb = local - c.mb * n_tiles;
  c.rows = seg_rows[c.g];
  return c;
}

// Shared-memory descriptor of an MN-major operand stored as MN blocks of 64 elements x
// the stage's K rows (128-byte swizzle): LBO = distance between the MN blocks, SBO =
// 1024 B between groups of 8 K rows.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t mn_block_bytes) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bwd(bool a_mn, int M) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// CG = 2: a CTA pair works one 256-row tile (dgrad: 256 rows of an expert segment; wgrad:
// 256 rows of the weight gradient); each CTA loads its own 128 rows of A and 128 of B's 256
// columns, the leader issues the pair MMAs (M = 256) and its commits reach both CTAs, and
// each CTA's epilogue drains its own TMEM rows.
template <int MODE, int CG>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_bwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB0x,
                       const __grid_constant__ CUtensorMap tmB1x, const BwdParams p) {
  using S = BwdSmem<CG>;
  constexpr int kStages = S::kStages, kBBytes = S::kBBytes, kStageBytes = S::kStageBytes;
  constexpr int TM = BM * CG;               // rows of a tile
  constexpr int kBoxes = (BN / CG) / 64;    // MN boxes of B per CTA
  constexpr bool kWgrad = MODE == WGRAD_DOWN || MODE == WGRAD_GU;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(bars + 32);
  int32_t* seg_rows = mt_prefix + kMaxGroups;
  uint8_t* sEpi = reinterpret_cast<uint8_t*>(seg_rows + kMaxGroups);  // [8 warps][32 rows][64 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.G + p.has_extra;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / CG, nunits = gridDim.x / CG;  // tile walkers (CTAs or pairs)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiWarps * CG);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
  }
  if (warp == 1) tmem_alloc_cg<CG>(tmem_slot, kTmemCols);
  if (warp == 2) build_tile_prefix(p.offsets, p.G, ngroups, p.T_extra, TM, lane, seg_rows, mt_prefix);
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = kWgrad ? ngroups * p.m_tiles_out * p.n_tiles : p.n_tiles * mt_prefix[ngroups];
  auto decode = [&](int tile) {
    return kWgrad ? decode_wgrad(tile, p.m_tiles_out, p.n_tiles, seg_rows)
                  : decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
  };
  auto kblocks_of = [&](const TileCoord& c) { return kWgrad ? (c.rows + BK - 1) / BK : p.K / BK; };
  auto group_row0 = [&](int g) { return g >= p.G ? p.a2_row_base : p.offsets[g]; };

  if (warp == 0) {
    // ======================= TMA producer (each CTA loads its own rows of A and half of B)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode(tile);
        const bool extra = c.g >= p.G;
        const int row0 = group_row0(c.g);
        const int kbs = kblocks_of(c);
        const int bx0 = c.nb * BN + (int)rank * (BN / CG);  // this CTA's first B column
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * kBBytes;
          const CUtensorMap* ta = &tmA;
          const CUtensorMap* tb;
          int ax, ay, by;
          bool a_two_boxes;
          if constexpr (kWgrad) {
            // A: activation [rows, M_out] MN-major; B: activation [rows, N_out] MN-major.
            // WGRAD_GU: A = dgu (padded rows), B = xd or x; WGRAD_DOWN: A = dyd, B = h (padded)
            const int y_pad = (int)padded_row0(row0, c.g) + kb * BK;
            ax = c.mb * TM + (int)rank * BM;
            ay = MODE == WGRAD_GU ? y_pad : row0 + kb * BK;
            a_two_boxes = true;
            tb = extra ? &tmB0x : &tmB0;
            by = MODE == WGRAD_DOWN ? (p.b_unpadded ? row0 + kb * BK : y_pad)
                                    : (extra ? p.extra_b_row0 + kb * BK : row0 + kb * BK);
          } else {
            // A: [rows, K] K-major, this CTA's 128 rows (dgu: padded rows); B: weight rows =
            // the K index, MN-major
            const int a_row0 = MODE == DGRAD_GU ? (int)padded_row0(row0, c.g) : row0;
            ax = kb * BK;
            ay = a_row0 + c.mb * TM + (int)rank * BM;
            a_two_boxes = false;
            if (MODE == DGRAD_DOWN || MODE == DGRAD_PLAIN) {
              tb = extra ? &tmB0x : &tmB0;
              by = kb * BK;
            } else {  // K = 2F: 128-column blocks alternate gate / up
              const bool up = (kb >> 1) & 1;
              tb = extra ? (up ? &tmB1x : &tmB0x) : (up ? &tmB1 : &tmB0);
              by = (kb >> 2) * 128 + (kb & 1) * 64;
            }
            by += extra ? 0 : c.g * p.b_group_rows;
          }
          if constexpr (CG == 1) {
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_2d(ta, a_dst, &full[stage], ax, ay);
            if (a_two_boxes) tma_load_2d(ta, a_dst + 8192, &full[stage], ax + 64, ay);
#pragma unroll
            for (int j = 0; j < kBoxes; ++j) tma_load_2d(tb, b_dst + 8192 * j, &full[stage], bx0 + 64 * j, by);
          } else {
            // both CTAs' loads complete on the leader's barrier, which expects both
            if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
            const uint32_t bar = mapa_shared(smem_addr(&full[stage]), 0);
            tma_load_2d_pair(ta, a_dst, bar, ax, ay);
            if (a_two_boxes) tma_load_2d_pair(ta, a_dst + 8192, bar, ax + 64, ay);
#pragma unroll
            for (int j = 0; j < kBoxes; ++j) tma_load_2d_pair(tb, b_dst + 8192 * j, bar, bx0 + 64 * j, by);
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      const int used = issued < kStages ? (int)issued : kStages;
      for (int i = 0; i < used; ++i) {
        const int s = (stage - 1 - i + 2 * kStages) % kStages;
        const uint32_t ph = (stage - 1 - i < 0) ? (phase ^ 1) : phase;
        if (ok) ok = mbar_wait(&empty[s], ph, abort, p.timeout_ns, p.status);
        if (!ok && (CG == 1 || leader)) mbar_wait_drain(&full[s], ph, p.timeout_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer (the leader of a pair issues for both CTAs)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bwd(kWgrad, TM);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode(tile);
        const int kbs = kblocks_of(c);
        if (kbs == 0) continue;  // an expert without rows: the epilogues write zeros
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort, p.timeout_ns, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < kbs; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = kWgrad ? desc_mn_sw128(a_addr + k * 2048, 8192) : desc_k_sw128(a_addr + k * 32);
            const uint64_t bd = desc_mn_sw128(b_addr + k * 2048, 8192);
            if constexpr (CG == 1) mma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0);
            else mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0);
          }
          if constexpr (CG == 1) mma_commit(&empty[stage]);
          else mma_commit_pair(&empty[stage], 0x3);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if constexpr (CG == 1) mma_commit(&tfull[acc]);
        else mma_commit_pair(&tfull[acc], 0x3);
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
      if constexpr (CG == 1) mma_commit(drain);
      else mma_commit_pair(drain, 0x3);
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    } else if (lane == 0 && CG == 2) {
      // the pair's MMAs write this CTA's TMEM and read its shared memory: stay until done
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ======================= epilogue (warps 2..9; TMEM lane quarter = warp % 4)
    const int quarter = warp & 3;
    const int cbase = ((warp - 2) >> 2) * (BN / 2);  // this warp's 128 of the tile's 256 columns
    const int wrow = (int)rank * BM + quarter * 32;   // the warp's first row in the tile
    const int r = wrow + lane;
    uint8_t* stage = sEpi + (warp - 2) * 2048;
    const uint32_t tempty_leader = CG == 2 ? mapa_shared(smem_addr(&tempty[0]), 0) : 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = unit; tile < total_tiles; tile += nunits) {
      const TileCoord c = decode(tile);
      const bool extra = c.g >= p.G;
      const bool empty_tile = kblocks_of(c) == 0;
      if (!empty_tile) {
        bool ok = mbar_wait(&tfull[acc], acc_phase, abort, p.timeout_ns, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if constexpr (kWgrad) {
        // fp32 gradient rows: row r of the output tile, 256 columns
        const int64_t ldo = p.N_out;
        float* wbase;
        if (MODE == WGRAD_DOWN) {
          wbase = (extra ? p.w0x : p.w0 + (int64_t)c.g * p.M_out * p.N_out) + ((int64_t)c.mb * TM + wrow) * ldo;
        } else {  // dgu's 128-row blocks alternate dWg / dWu rows of one F block
          const int blk = c.mb * CG + (int)rank;
          const bool up = blk & 1;
          float* w = up ? (extra ? p.w1x : p.w1 + (int64_t)c.g * p.F * p.N_out)
                        : (extra ? p.w0x : p.w0 + (int64_t)c.g * p.F * p.N_out);
          wbase = w + ((int64_t)(blk >> 1) * BM + quarter * 32) * ldo;
        }
        uint8_t* out = reinterpret_cast<uint8_t*>(wbase + c.nb * BN + cbase);
        uint32_t nxt[32];
        if (!empty_tile) tmem_ld32(t_row + cbase, nxt);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t v[32];
          if (!empty_tile) {
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = nxt[i];
            if (c0 + 32 < BN / 2) tmem_ld32(t_row + cbase + c0 + 32, nxt);  // next chunk in flight
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {  // 16 fp32 = 64 bytes per pass
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece(stage, lane, q, make_uint4(v[16 * h2 + 4 * q], v[16 * h2 + 4 * q + 1], v[16 * h2 + 4 * q + 2],
                                                     v[16 * h2 + 4 * q + 3]));
            flush_rows_64B(stage, lane, out + 4 * (c0 + 16 * h2), ldo * 4, 32);
          }
        }
      } else {
        const int row0 = group_row0(c.g);
        const int64_t warp_row0 = (int64_t)row0 + c.mb * TM + wrow;
        const int warp_live = c.rows - wrow;
        const bool live = r < c.rows;
        if (MODE == DGRAD_GU || MODE == DGRAD_PLAIN) {
          uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + (warp_row0 * p.ldc + c.nb * BN + cbase) * 2;
#pragma unroll 1
          for (int c0 = 0; c0 < BN / 2; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(t_row + cbase + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece(stage, lane, q,
                          make_uint4(pack_bf16(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                                     pack_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                     pack_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                     pack_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]))));
            flush_rows_64B(stage, lane, out + 2 * c0, (int64_t)p.ldc * 2, warp_live);
          }
        } else {  // DGRAD_DOWN: dh -> SwiGLU backward with g, u from gu; writes dg, du and h
          const int64_t row = warp_row0 + lane;
          const int ld_gu = 2 * p.F;
          // dgu and h rows are padded: this warp's rows start at prow0, and the rows past the
          // segment up to its multiple of 64 are written as zeros (g = u = 0 there)
          const int64_t prow0 = padded_row0(row0, c.g) + c.mb * TM + wrow;
          const int seg = c.g < p.G ? p.offsets[c.g + 1] - p.offsets[c.g] : p.T_extra;
          const int pad_live = min((seg + 63) / 64 * 64 - c.mb * TM, TM) - wrow;
#pragma unroll 1
          for (int c0 = cbase; c0 < cbase + BN / 2; c0 += 32) {
            const int f0 = c.nb * BN + c0;     // first F column of the chunk
            const int blk = f0 >> 7, cb = f0 & 127;
            uint32_t dh[32];
            tmem_ld32(t_row + c0, dh);
            uint4 graw[4], uraw[4];
            if (live) {
              const uint4* gp = reinterpret_cast<const uint4*>(p.gu + row * ld_gu + blk * 256 + cb);
              const uint4* up = reinterpret_cast<const uint4*>(p.gu + row * ld_gu + blk * 256 + 128 + cb);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                graw[q] = __ldg(gp + q);
                uraw[q] = __ldg(up + q);
              }
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) graw[q] = uraw[q] = make_uint4(0, 0, 0, 0);
            }
            tmem_ld_wait();
            uint32_t pdg[16], pdu[16], ph[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t gw[4] = {graw[q].x, graw[q].y, graw[q].z, graw[q].w};
              const uint32_t uw[4] = {uraw[q].x, uraw[q].y, uraw[q].z, uraw[q].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float dgv[2], duv[2], hv[2];
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                  const float g = __uint_as_float(s2 ? (gw[e] & 0xffff0000u) : (gw[e] << 16));
                  const float u = __uint_as_float(s2 ? (uw[e] & 0xffff0000u) : (uw[e] << 16));
                  const float d = __uint_as_float(dh[8 * q + 2 * e + s2]);
                  const float sg = 1.0f / (1.0f + __expf(-g));
                  const float silu = g * sg;
                  hv[s2] = silu * u;
                  dgv[s2] = d * u * sg * (1.0f + g * (1.0f - sg));
                  duv[s2] = d * silu;
                }
                pdg[4 * q + e] = pack_bf16(dgv[0], dgv[1]);
                pdu[4 * q + e] = pack_bf16(duv[0], duv[1]);
                ph[4 * q + e] = pack_bf16(hv[0], hv[1]);
              }
            }
            uint8_t* dgu_rows = reinterpret_cast<uint8_t*>(p.out) + (prow0 * ld_gu + blk * 256 + cb) * 2;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece(stage, lane, q, make_uint4(pdg[4 * q], pdg[4 * q + 1], pdg[4 * q + 2], pdg[4 * q + 3]));
            flush_rows_64B(stage, lane, dgu_rows, (int64_t)ld_gu * 2, pad_live);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece(stage, lane, q, make_uint4(pdu[4 * q], pdu[4 * q + 1], pdu[4 * q + 2], pdu[4 * q + 3]));
            flush_rows_64B(stage, lane, dgu_rows + 256, (int64_t)ld_gu * 2, pad_live);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              stage_piece(stage, lane, q, make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]));
            flush_rows_64B(stage, lane, reinterpret_cast<uint8_t*>(p.h_out) + (prow0 * p.F + f0) * 2,
                           (int64_t)p.F * 2, pad_live);
          }
        }
      }
      if (!empty_tile) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2 && !leader) mbar_arrive_cluster_relaxed(tempty_leader + acc * 8);
          else mbar_arrive_relaxed(&tempty[acc]);
        }
        if (++acc == 2) { acc = 0; acc_phase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // neither CTA leaves while the pair still uses it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_cg<CG>(tmem_base, kTmemCols);
  }
}

bool make_bf16_box(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, box_rows, 64);
}

template <int MODE, int CG>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b0x,
                   const CUtensorMap& b1x, const BwdParams& p, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  auto kern = tc_gemm_bwd_kernel<MODE, CG>;
  const size_t smem = BwdSmem<CG>::kBytes;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if constexpr (CG == 1) {
    const int grid = (int)std::min<int64_t>(num_sms(), max_tiles);
    kern<<<grid, kThreads, smem, s>>>(a, b0, b1, b0x, b1x, p);
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a, b0, b1, b0x, b1x, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

int64_t backward_padded_rows(const moe_config_t& c) {
  return total_rows(c) + 63 * ((int64_t)c.E + 1) + 64;
}

bool mlp_backward_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.xfer_dtype == MOE_DTYPE_BF16 && c.H % 256 == 0 && c.F % 256 == 0 &&
         c.E + 1 <= kMaxGroups;
}

cudaError_t launch_grouped_mlp_backward(const moe_config_t& c, const void* xd, const void* x,
                                        const int32_t* offsets, const moe_weights_t& w, const void* dyd, void* gu,
                                        void* dgu, void* h, void* dxd, const moe_weight_grads_t& gr,
                                        DeviceStatus* st, cudaStream_t s, bool gu_ready) {
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  const int64_t prows = backward_padded_rows(c);  // rows of the padded dgu and h
  // dgrad tiles are expert segments: CTA pairs (256-row tiles) when experts average at least
  // 512 rows, as in the forward; wgrad tiles are weight-gradient rows and always pairs
  const bool pair = (int64_t)c.T * c.k >= 512LL * c.E;
  const int tm = pair ? 2 * BM : BM;
  const int64_t mt_bound = ceil_div(R, tm) + c.E + (shared ? ceil_div(c.T, tm) : 0);
  // ---- recompute g and u (the forward GEMM1 without its activation), unless kept
  cudaError_t e = gu_ready ? cudaSuccess : launch_gate_up_preact(c, xd, x, offsets, w, gu, st, s);
  if (e != cudaSuccess) return e;
  BwdParams p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = (int)R;
  p.F = c.F;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  // ---- dh = dyd Wd, then dg, du, h (B = Wd [E*H rows, F cols] read MN-major)
  CUtensorMap a, b0, b1, b0x, b1x;
  bool ok = make_bf16_box(&a, dyd, rows, c.H, BM) && make_bf16_box(&b0, w.w_down, (uint64_t)c.E * c.H, c.F, 64);
  if (shared) ok = ok && make_bf16_box(&b0x, w.ws_down, c.H, c.F, 64);
  else b0x = b0;
  if (!ok) return cudaErrorInvalidValue;
  p.K = c.H;
  p.n_tiles = c.F / BN;
  p.b_group_rows = c.H;
  p.ldc = 2 * c.F;
  p.out = static_cast<__nv_bfloat16*>(dgu);
  p.h_out = static_cast<__nv_bfloat16*>(h);
  p.gu = static_cast<const __nv_bfloat16*>(gu);
  e = pair ? launch<DGRAD_DOWN, 2>(a, b0, b0, b0x, b0x, p, mt_bound * p.n_tiles, s)
           : launch<DGRAD_DOWN, 1>(a, b0, b0, b0x, b0x, p, mt_bound * p.n_tiles, s);
  if (e != cudaSuccess) return e;
  // ---- dxd = dg Wg + du Wu (K = 2F in dgu's interleaved order; B = Wg or Wu rows)
  ok = make_bf16_box(&a, dgu, prows, 2 * (uint64_t)c.F, BM) && make_bf16_box(&b0, w.w_gate, (uint64_t)c.E * c.F, c.H, 64) &&
       make_bf16_box(&b1, w.w_up, (uint64_t)c.E * c.F, c.H, 64);
  if (shared) ok = ok && make_bf16_box(&b0x, w.ws_gate, c.F, c.H, 64) && make_bf16_box(&b1x, w.ws_up, c.F, c.H, 64);
  else { b0x = b0; b1x = b1; }
  if (!ok) return cudaErrorInvalidValue;
  p.K = 2 * c.F;
  p.n_tiles = c.H / BN;
  p.b_group_rows = c.F;
  p.ldc = c.H;
  p.out = static_cast<__nv_bfloat16*>(dxd);
  e = pair ? launch<DGRAD_GU, 2>(a, b0, b1, b0x, b1x, p, mt_bound * p.n_tiles, s)
           : launch<DGRAD_GU, 1>(a, b0, b1, b0x, b1x, p, mt_bound * p.n_tiles, s);
  if (e != cudaSuccess) return e;
  // ---- dWd[e] = dyd_e^T h_e (M_out = H, N_out = F; both operands MN-major)
  const int ngroups = c.E + (shared ? 1 : 0);
  ok = make_bf16_box(&a, dyd, rows, c.H, 64) && make_bf16_box(&b0, h, prows, c.F, 64);
  if (!ok) return cudaErrorInvalidValue;
  p.extra_b_row0 = 0;  // unused: h's rows are addressed by their padded position
  p.M_out = c.H;
  p.N_out = c.F;
  p.m_tiles_out = c.H / (2 * BM);
  p.n_tiles = c.F / BN;
  p.w0 = gr.dw_down;
  p.w0x = gr.dws_down;
  p.w1 = p.w1x = nullptr;
  e = launch<WGRAD_DOWN, 2>(a, b0, b0, b0, b0, p, (int64_t)ngroups * p.m_tiles_out * p.n_tiles, s);
  if (e != cudaSuccess) return e;
  // ---- dWg[e], dWu[e] = dgu_e^T xd_e (M_out = 2F interleaved, N_out = H)
  // xd's map ends at the last routed row: the TMA fills zeros past it, never reading rows
  // the dispatch did not write
  ok = make_bf16_box(&a, dgu, prows, 2 * (uint64_t)c.F, 64) && make_bf16_box(&b0, xd, R, c.H, 64);
  if (shared) ok = ok && make_bf16_box(&b0x, x, c.T, c.H, 64);  // the shared expert's input is x
  else b0x = b0;
  if (!ok) return cudaErrorInvalidValue;
  p.extra_b_row0 = 0;
  p.M_out = 2 * c.F;
  p.N_out = c.H;
  p.m_tiles_out = 2 * c.F / (2 * BM);
  p.n_tiles = c.H / BN;
  p.w0 = gr.dw_gate;
  p.w1 = gr.dw_up;
  p.w0x = gr.dws_gate;
  p.w1x = gr.dws_up;
  return launch<WGRAD_GU, 2>(a, b0, b0, b0x, b0x, p, (int64_t)ngroups * p.m_tiles_out * p.n_tiles, s);
}

bool router_backward_tc_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.E % 128 == 0 && c.H % 256 == 0;
}

cudaError_t launch_router_products(const moe_config_t& c, const void* dl_bf16, const void* x, const void* w_router,
                                   float* dw_router, void* dx_r, DeviceStatus* st, cudaStream_t s,
                                   const int32_t* slice_offsets, int slices) {
  if (c.T == 0) return cudaSuccess;
  // the tokens are one group: the "extra" group of the kernels (no routed groups), rows [0, T)
  BwdParams p{};
  p.offsets = nullptr;
  p.G = 0;
  p.has_extra = 1;
  p.T_extra = c.T;
  p.a2_row_base = 0;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  CUtensorMap a, b;
  cudaError_t e = cudaSuccess;
  if (dw_router) {
    // dW_router = dl^T x: M_out = E, N_out = H, K = T, both operands MN-major; the maps end
    // at row T, so the last K stage reads zeros past it
    if (!make_bf16_box(&a, dl_bf16, c.T, c.E, 64) || !make_bf16_box(&b, x, c.T, c.H, 64)) return cudaErrorInvalidValue;
    // 256-row tiles as CTA pairs when E allows, else 128-row tiles on single CTAs. With
    // slices > 1 the tokens are split into that many groups (K splits, slice_offsets on the
    // device, whole 64-row stages but the last): dw_router then receives the per-slice
    // partial sums [slices, E, H], which the caller adds in slice order.
    const bool pair = c.E % 256 == 0;
    p.M_out = c.E;
    p.N_out = c.H;
    p.m_tiles_out = c.E / (pair ? 2 * BM : BM);
    p.n_tiles = c.H / BN;
    p.w0 = nullptr;
    p.w0x = dw_router;
    if (slices > 1) {
      p.offsets = slice_offsets;
      p.G = slices;
      p.has_extra = 0;
      p.T_extra = 0;
      p.w0 = dw_router;
      p.w0x = nullptr;
      p.b_unpadded = 1;
    }
    const int64_t tiles = (int64_t)(p.G + p.has_extra) * p.m_tiles_out * p.n_tiles;
    e = pair ? launch<WGRAD_DOWN, 2>(a, b, b, b, b, p, tiles, s) : launch<WGRAD_DOWN, 1>(a, b, b, b, b, p, tiles, s);
    if (e != cudaSuccess) return e;
    p.offsets = nullptr;
    p.G = 0;
    p.has_extra = 1;
    p.T_extra = c.T;
    p.b_unpadded = 0;
  }
  if (dx_r) {
    // dx_r = dl W_router: M = T, N = H, K = E; W_router [E, H] read MN-major
    if (!make_bf16_box(&a, dl_bf16, c.T, c.E, BM) || !make_bf16_box(&b, w_router, c.E, c.H, 64))
      return cudaErrorInvalidValue;
    const bool pair = c.T >= 512;
    const int tm = pair ? 2 * BM : BM;
    p.K = c.E;
    p.n_tiles = c.H / BN;
    p.b_group_rows = 0;
    p.ldc = c.H;
    p.out = static_cast<__nv_bfloat16*>(dx_r);
    const int64_t tiles = ceil_div(c.T, tm) * p.n_tiles;
    e = pair ? launch<DGRAD_PLAIN, 2>(a, b, b, b, b, p, tiles, s) : launch<DGRAD_PLAIN, 1>(a, b, b, b, b, p, tiles, s);
  }
  return e;
}

}  // namespace tc
}  // namespace moe
