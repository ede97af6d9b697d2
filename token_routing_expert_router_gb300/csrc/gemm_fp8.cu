// FP8 (e4m3) grouped expert GEMMs with fp32 block scales, on the tcgen05 tensor cores.
//
// The FP8-dispatch variant quantises tokens in 1x128 blocks and weights in 128x128 blocks
// with fp32 scales that are not powers of two ("Scalable Training of Mixture-of-Experts
// Models with Megatron Core" summary, FP8/FP4 reduced precision; the Hybrid-EP article,
// low-precision dispatch). The hardware's block-scaled MMA takes only power-of-two scales,
// so the scales are applied in software: every 128-wide K block is accumulated by
// tcgen05.mma (kind::f8f6f4, e4m3 x e4m3 -> fp32) into one of two TMEM partial buffers,
// and the epilogue warps add sa[row, kb] * sb[n-block, kb] * partial into fp32 registers
// while the tensor core fills the other buffer.
//
// Block: warp 0 TMA producer, warp 1 MMA issuer (TMEM owner), warps 2-9 epilogue: two
// warps per TMEM lane quarter, each owning half of the tile's 256 columns.
//   GEMM1 (gate/up): columns [0,128) gate and [128,256) up of one 128-wide F block; a
//     thread owns 64 gate + 64 up columns, computes h = silu(g) * u, and the row's 128 h
//     values are requantised to e4m3 in one 1x128 block (amax shared through smem).
//   GEMM2 (down): 256 output columns = two 128-row weight scale blocks; bf16 output.
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "tc_common.cuh"

namespace moe {
namespace tc {

bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols);
int num_sms();

namespace {

constexpr int BM = 128, BN = 256, BK = 128;  // BK in elements = bytes (e4m3)
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kMaxGroups = 514;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kABytes = BM * BK;
constexpr int kTmemCols = 512;  // two 256-column partial accumulators

// Shared memory of one CTA: four 48 KB stages (A 16 KB + B 32 KB).
struct F8Smem {
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 4;
  static constexpr size_t kBytes = 1024 + (size_t)kStages * kStageBytes + 256 + 2 * BM * sizeof(float) +
                                   2 * kMaxGroups * sizeof(int32_t) + (kEpiThreads / 32) * 2048 /*store staging*/;
};

enum { FP8_SWIGLU_Q8 = 0, FP8_STORE_BF16 = 1 };

struct Fp8Params {
  const int32_t* offsets;
  int G, has_extra, T_extra, a2_row_base;
  int64_t out_extra_base;
  int K;             // multiple of 128
  int n_tiles;       // N tiles of 256 columns per group (GEMM1: F/128; GEMM2: N/256)
  int b_group_rows;  // rows of B per routed group
  int64_t rows_total;      // rows of A (and of its scale matrix)
  const float* a_scale;    // [K/128][rows_total]
  const float* b0_scale;   // routed: GEMM1 gate [G, F/128, K/128]; GEMM2 [G, N/128, K/128]
  const float* b1_scale;   // routed: GEMM1 up
  const float* b0x_scale;  // extra group's
  const float* b1x_scale;
  int nblk_b;              // 128-row blocks of B per group (F/128 or N/128)
  int ldc;                 // output row length (elements)
  void* out;               // GEMM1: h e4m3 [rows, F]; GEMM2: yd bf16 [rows, N]
  float* out_scale;        // GEMM1: h_scale [F/128][rows_total]
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// TMEM column of the q-th 16-column chunk a thread of column-half `half` promotes.
// GEMM1: q 0-3 gate cols [half*64, +64), q 4-7 up cols [128 + half*64, +64);
// GEMM2: cols [half*128 + 16q, +16).
template <int EPI>
__device__ __forceinline__ uint32_t col_of_t(int q, int half) {
  return EPI == 0 ? (q < 4 ? half * 64 + 16 * q : 128 + half * 64 + 16 * (q - 4)) : half * 128 + 16 * q;
}

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ CUtensorMap tmB0x, const __grid_constant__ CUtensorMap tmB1x,
                       const Fp8Params p) {
  using S = F8Smem;
  constexpr int kStages = S::kStages, kBBytes = S::kBBytes, kStageBytes = S::kStageBytes;
  constexpr int TM = BM;  // rows of an m tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* pfull = bars + 2 * kStages;  // [2] partial accumulator ready
  uint64_t* pempty = pfull + 2;          // [2] partial accumulator read by the epilogue
  uint64_t* drain = pempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* amax_buf = reinterpret_cast<float*>(bars + 32);  // [2][BM]
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(amax_buf + 2 * BM);
  int32_t* seg_rows = mt_prefix + kMaxGroups;
  uint8_t* sEpi = reinterpret_cast<uint8_t*>(seg_rows + kMaxGroups);  // [8 warps][32 rows][64 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.G + p.has_extra;
  auto col_of = [](int q, int half) { return col_of_t<EPI>(q, half); };
  const int unit = blockIdx.x, nunits = gridDim.x;  // persistent tile walkers

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&pfull[a], 1);
      mbar_init(&pempty[a], kEpiThreads / 32);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
  }
  if (warp == 1) tmem_alloc_cg<1>(tmem_slot, kTmemCols);
  if (warp == 2) build_tile_prefix(p.offsets, p.G, ngroups, p.T_extra, TM, lane, seg_rows, mt_prefix);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.n_tiles * mt_prefix[ngroups];
  const int kblocks = p.K / BK;

  if (warp == 0) {
    // ======================= TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
        const bool extra = c.g >= p.G;
        const CUtensorMap* ta = extra ? &tmA2 : &tmA;
        const CUtensorMap* tb0 = extra ? &tmB0x : &tmB0;
        const CUtensorMap* tb1 = extra ? &tmB1x : &tmB1;
        const int a_row = (extra ? p.a2_row_base : p.offsets[c.g]) + c.mb * TM;
        const int b_tile_rows = EPI == FP8_SWIGLU_Q8 ? BN / 2 : BN;
        const int b_row = (extra ? 0 : c.g * p.b_group_rows) + c.nb * b_tile_rows;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * kBBytes;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tma_load_2d(ta, a_dst, &full[stage], kb * BK, a_row);
          if (EPI == FP8_SWIGLU_Q8) {
            tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);
            tma_load_2d(tb1, b_dst + (BN / 2) * BK, &full[stage], kb * BK, b_row);
          } else {
            tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);
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
        if (!ok) mbar_wait_drain(&full[s], ph, p.timeout_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer: one partial accumulator per K block
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_make(0u /*e4m3*/, TM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int pb = 0;
      uint32_t pphase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&pempty[pb], pphase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
          if (!mbar_wait(&full[stage], phase, abort, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kBBytes);
          const uint32_t d_tmem = tmem_base + pb * BN;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // K = 32 e4m3 per instruction: +32 bytes
            mma_f8(d_tmem, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + k * 32), idesc, k != 0);
          mma_commit(&empty[stage]);
          mma_commit(&pfull[pb]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          if (++pb == 2) { pb = 0; pphase ^= 1; }
        }
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ======================= epilogue: warps 2..9
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;  // which 128 of the 256 tile columns this warp owns
    const int r = quarter * 32 + lane;
    int pb = 0;
    uint32_t pphase = 0;
    int tile_parity = 0;
    bool ok = true;
    for (int tile = unit; tile < total_tiles; tile += nunits, tile_parity ^= 1) {
      const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
      const bool extra = c.g >= p.G;
      const int row_in_tile = r;
      const int64_t a_row = (extra ? (int64_t)p.a2_row_base : (int64_t)p.offsets[c.g]) + c.mb * TM + row_in_tile;
      const int64_t a_row_c = a_row < p.rows_total ? a_row : p.rows_total - 1;  // dead rows: any scale
      const float* sb0 = (extra ? p.b0x_scale : p.b0_scale + (int64_t)c.g * p.nblk_b * kblocks);
      const float* sb1 = (extra ? p.b1x_scale : p.b1_scale + (int64_t)c.g * p.nblk_b * kblocks);
      // scale rows of this tile's weight blocks
      const float* sbA;  // columns [0, 64) of this thread's 128 (GEMM1: gate; GEMM2: block 2nb+half)
      const float* sbB;  // columns [64, 128)           (GEMM1: up)
      if (EPI == FP8_SWIGLU_Q8) {
        sbA = sb0 + (int64_t)c.nb * kblocks;
        sbB = sb1 + (int64_t)c.nb * kblocks;
      } else {
        sbA = sb0 + (int64_t)(2 * c.nb + half) * kblocks;
        sbB = sbA;
      }
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      float sa_next = p.a_scale[a_row_c];
      float sbA_next = sbA[0], sbB_next = sbB[0];
      for (int kb = 0; kb < kblocks; ++kb) {
        const float sa = sa_next, fa = sa * sbA_next, fb = sa * sbB_next;
        if (kb + 1 < kblocks) {  // next block's scales load while this one is waited for
          sa_next = p.a_scale[(int64_t)(kb + 1) * p.rows_total + a_row_c];
          sbA_next = sbA[kb + 1];
          sbB_next = sbB[kb + 1];
        }
        // After an abort the warp keeps walking the same tiles without waiting or loading,
        // so that every epilogue warp still reaches each named barrier below.
        if (ok) ok = mbar_wait(&pfull[pb], pphase, abort, p.timeout_ns, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          const uint32_t t = tmem_base + ((uint32_t)(quarter * 32) << 16) + pb * BN;
          // software-pipelined: the load of chunk q + 1 is in flight while chunk q's FMAs run
          uint32_t v[2][16];
          tmem_ld16(t + col_of(0, half), v[0]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q < 7) tmem_ld16(t + col_of(q + 1, half), v[(q + 1) & 1]);
            const float f = (q < 4) ? fa : fb;
#pragma unroll
            for (int i = 0; i < 16; i += 2)
              fma2(acc[16 * q + i], acc[16 * q + i + 1], __uint_as_float(v[q & 1][i]),
                   __uint_as_float(v[q & 1][i + 1]), f);
            tmem_ld_wait();
            if (q == 6) {  // every chunk of this buffer has been read: hand it back to the MMA
              tc_fence_before();
              __syncwarp();    // all lanes' loads are complete: one arrival per warp
              if (lane == 0) mbar_arrive_relaxed(&pempty[pb]);
            }
          }
        }
        if (++pb == 2) { pb = 0; pphase ^= 1; }
      }
      const int64_t out_row = (extra ? p.out_extra_base : (int64_t)p.offsets[c.g]) + c.mb * TM + row_in_tile;
      const bool live = ok && row_in_tile < c.rows;
      if (EPI == FP8_SWIGLU_Q8) {
        // h = silu(g) * u for this thread's 64 columns; 1x128 requantisation across both halves
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float g = acc[i];
          const float h = g / (1.0f + __expf(-g)) * acc[64 + i];
          acc[i] = h;
          amax = fmaxf(amax, fabsf(h));
        }
        float* ab = amax_buf + tile_parity * BM;
        if (half == 1) ab[r] = amax;
        epi_bar_sync();
        if (half == 0) ab[r] = fmaxf(ab[r], amax);
        epi_bar_sync();
        amax = ab[r];
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        const float rs = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 0.0f;
        if (live) {
          uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + out_row * p.ldc + c.nb * 128 + half * 64;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 o;
            o.x = e4m3x4(__fmul_rn(acc[16 * q + 0], rs), __fmul_rn(acc[16 * q + 1], rs), __fmul_rn(acc[16 * q + 2], rs), __fmul_rn(acc[16 * q + 3], rs));
            o.y = e4m3x4(__fmul_rn(acc[16 * q + 4], rs), __fmul_rn(acc[16 * q + 5], rs), __fmul_rn(acc[16 * q + 6], rs), __fmul_rn(acc[16 * q + 7], rs));
            o.z = e4m3x4(__fmul_rn(acc[16 * q + 8], rs), __fmul_rn(acc[16 * q + 9], rs), __fmul_rn(acc[16 * q + 10], rs), __fmul_rn(acc[16 * q + 11], rs));
            o.w = e4m3x4(__fmul_rn(acc[16 * q + 12], rs), __fmul_rn(acc[16 * q + 13], rs), __fmul_rn(acc[16 * q + 14], rs), __fmul_rn(acc[16 * q + 15], rs));
            reinterpret_cast<uint4*>(out)[q] = o;
          }
          if (half == 0) p.out_scale[(int64_t)c.nb * p.rows_total + out_row] = scale;
        }
      } else {
        // bf16 rows leave through a per-warp shared-memory staging buffer, 32 columns at a
        // time, so that each store instruction writes 8 rows x 64 contiguous bytes
        uint8_t* stage = sEpi + ew * 2048;
        const int warp_live = ok ? c.rows - (row_in_tile - lane) : 0;
        uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + ((out_row - lane) * p.ldc + c.nb * BN + half * 128) * 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t w4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = 32 * q + 8 * c4 + 2 * j;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[i], acc[i + 1]);
              w4[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            stage_piece(stage, lane, c4, make_uint4(w4[0], w4[1], w4[2], w4[3]));
          }
          flush_rows_64B(stage, lane, out + 64 * q, (int64_t)p.ldc * 2, warp_live);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_cg<1>(tmem_base, kTmemCols);
  }
}

bool make_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return make_tmap(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, box_rows, BK);
}

template <int EPI>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b0, const CUtensorMap& b1,
                   const CUtensorMap& b0x, const CUtensorMap& b1x, const Fp8Params& p, int64_t max_tiles,
                   cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  auto kern = tc_gemm_fp8_kernel<EPI>;
  const size_t smem = F8Smem::kBytes;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = (int)std::min<int64_t>(num_sms(), max_tiles);
  kern<<<grid, kThreads, smem, s>>>(a, a2, b0, b1, b0x, b1x, p);
  return cudaGetLastError();
}

}  // namespace

bool fp8_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.xfer_dtype == MOE_DTYPE_E4M3 && c.H % 256 == 0 && c.F % 128 == 0;
}

cudaError_t launch_grouped_mlp_fp8(const moe_config_t& c, const void* xd, const float* xd_scale,
                                   const int32_t* offsets, const moe_weights_t& w, void* h, float* h_scale,
                                   void* yd, DeviceStatus* st, cudaStream_t s) {
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  // ---- GEMM1: h = e4m3(silu(A Wg^T) * (A Wu^T)), the shared expert's A = dispatched rows R..
  CUtensorMap a1, bg, bu, bgx, bux;
  bool ok = make_u8(&a1, xd, rows, c.H, BM) && make_u8(&bg, w.w_gate, (uint64_t)c.E * c.F, c.H, 128) &&
            make_u8(&bu, w.w_up, (uint64_t)c.E * c.F, c.H, 128);
  if (shared) ok = ok && make_u8(&bgx, w.ws_gate, c.F, c.H, 128) && make_u8(&bux, w.ws_up, c.F, c.H, 128);
  else { bgx = bg; bux = bu; }
  if (!ok) return cudaErrorInvalidValue;
  Fp8Params p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = (int)R;
  p.out_extra_base = R;
  p.K = c.H;
  p.n_tiles = c.F / 128;
  p.b_group_rows = c.F;
  p.rows_total = rows;
  p.a_scale = xd_scale;
  p.b0_scale = static_cast<const float*>(w.s_gate);
  p.b1_scale = static_cast<const float*>(w.s_up);
  p.b0x_scale = static_cast<const float*>(shared ? w.ss_gate : w.s_gate);
  p.b1x_scale = static_cast<const float*>(shared ? w.ss_up : w.s_up);
  p.nblk_b = c.F / 128;
  p.ldc = c.F;
  p.out = h;
  p.out_scale = h_scale;
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  // Single-CTA tiles: a CTA-pair form of this kernel computed the same results but ran at
  // half the rate, because the partial accumulator it hands from the MMA to the epilogue
  // every K block then crosses SMs with only two partial buffers to hide the handshake.
  const int64_t mt_bound = ceil_div(R, BM) + c.E + (shared ? ceil_div(c.T, BM) : 0);
  cudaError_t e = launch<FP8_SWIGLU_Q8>(a1, a1, bg, bu, bgx, bux, p, mt_bound * p.n_tiles, s);
  if (e != cudaSuccess) return e;
  // ---- GEMM2: yd = (h * h_scale) (Wd * s_down)^T, bf16 out
  CUtensorMap a2, bd, bdx;
  ok = make_u8(&a2, h, rows, c.F, BM) && make_u8(&bd, w.w_down, (uint64_t)c.E * c.H, c.F, BN);
  if (shared) ok = ok && make_u8(&bdx, w.ws_down, c.H, c.F, BN);
  else bdx = bd;
  if (!ok) return cudaErrorInvalidValue;
  p.K = c.F;
  p.n_tiles = c.H / BN;
  p.b_group_rows = c.H;
  p.a_scale = h_scale;
  p.b0_scale = static_cast<const float*>(w.s_down);
  p.b1_scale = p.b0_scale;
  p.b0x_scale = static_cast<const float*>(shared ? w.ss_down : w.s_down);
  p.b1x_scale = p.b0x_scale;
  p.nblk_b = c.H / 128;
  p.ldc = c.H;
  p.out = yd;
  p.out_scale = nullptr;
  return launch<FP8_STORE_BF16>(a2, a2, bd, bd, bdx, bdx, p, mt_bound * p.n_tiles, s);
}

}  // namespace tc
}  // namespace moe
