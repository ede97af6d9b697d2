// MXFP8 grouped expert GEMMs on the block-scaled tcgen05 tensor-core MMA.
//
// The MXFP8 variant ("Scalable Training of Mixture-of-Experts Models with Megatron Core"
// summary, reduced precision on Blackwell; the Hybrid-EP article's MXFP8 results) carries
// one power-of-two UE8M0 scale per 1x32 block of every operand row (OCP MX v1.0). Such
// scales are applied by the tensor core itself: tcgen05.mma.kind::mxf8f6f4.block_scale
// multiplies each 32-wide K slice of A and B by their scale factors, which it reads from
// tensor memory, so the whole K loop accumulates in one TMEM accumulator with no software
// promotion.
//
// Tile 128 x 256 (one CTA), K stages of 128 (four MMAs of K = 32, scale-factor id = the
// slice).
// Block: warp 0 TMA producer, warp 1 MMA issuer (TMEM owner), warps 2-9 epilogue (two
// warps per TMEM lane quarter, each owning half of the tile's columns).
//   Per stage the producer loads the A and B tiles (TMA, 128-byte swizzle) and the stage's
//   scale atoms (one 512-byte atom per 128 rows, TMA boxes of a linear [atoms, 128 x u32]
//   view); the MMA issuer moves the atoms into tensor memory with tcgen05.cp 32x128b.warpx4
//   (the copy and the MMAs that read it come from one thread, so they execute in order)
//   and issues the MMAs.
//   TMEM: accumulator in columns [0, 256); stage s's scale factors in [256 + 16s, +12).
//   The accumulator is single-buffered: the epilogue loads its 128 x 256 values into
//   registers and hands the accumulator back before it computes and stores, so the next
//   tile's MMAs wait only for the loads.
//   GEMM1 (gate/up): columns [0,128) gate and [128,256) up of one 128-wide F block; a
//     thread owns 64 gate + 64 up columns of one row, computes h = silu(g) * u and
//     requantises its two 1x32 blocks of h (the scale is thread-local), writing h's codes
//     and its UE8M0 codes into h's scale atoms.
//   GEMM2 (down): 256 output columns, bf16, stored through a per-warp shared-memory
//     staging buffer (the row-per-thread TMEM layout would otherwise make every store
//     instruction touch 32 rows).
#include <cudaTypedefs.h>

#include "gemm_tc.cuh"
#include "mx_common.cuh"
#include "tc_common.cuh"

namespace moe {
namespace tc {

bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows, uint64_t cols,
               uint32_t box_rows, uint32_t box_cols);
bool make_tmap_linear(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t rows,
                      uint64_t cols, uint32_t box_rows, uint32_t box_cols);
int num_sms();

namespace {

constexpr int BM = 128, BN = 256, BK = 128;  // BK in elements = bytes (e4m3)
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kABytes = BM * BK;
constexpr int kAtomBytes = 512;
constexpr int kSfBytes = 3 * kAtomBytes;  // A atom, then B atoms for columns [0,128), [128,256)
constexpr int kMaxGroups = 514;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kTmemCols = 512;
constexpr uint32_t kSfCol0 = 256, kSfColsPerStage = 16;  // up to 6 stages: columns 256..351
constexpr int kEpiStageBytes = 32 * 64;  // per epilogue warp: 32 rows x 64 bytes (GEMM2 stores)

struct MxSmem {
  static constexpr int kBBytes = BN * BK;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;
  static constexpr int kStages = 4;
  static constexpr size_t kBytes = 1024 + (size_t)kStages * kStageBytes + 256 + 2 * kMaxGroups * sizeof(int32_t) +
                                   kEpiWarps * kEpiStageBytes;
};

enum { MX_SWIGLU_Q8 = 0, MX_STORE_BF16 = 1 };

struct MxParams {
  const int32_t* offsets;
  int G, has_extra, T_extra, a2_row_base;  // the extra (shared) group's A rows start at a2_row_base = T*k
  int64_t out_extra_base;
  int K;             // multiple of 128
  int n_tiles;       // N tiles per group (GEMM1: F/128; GEMM2: N/256)
  int b_group_rows;  // rows of B per routed group (GEMM1: F; GEMM2: N)
  const uint8_t* a_sf;    // A's scale atoms, grouped rows (K columns)
  const uint8_t* b0_sf;   // routed weights' atoms: GEMM1 gate [G*F/128][K/128]; GEMM2 down [G*N/128][K/128]
  const uint8_t* b1_sf;   // GEMM1 up
  const uint8_t* b0x_sf;  // the shared expert's
  const uint8_t* b1x_sf;
  int ldc;                // output row length (elements)
  void* out;              // GEMM1: h e4m3 [rows, F]; GEMM2: yd bf16 [rows, N]
  uint8_t* out_sf;        // GEMM1: h's scale atoms (F columns)
  DeviceStatus* status;
  uint64_t timeout_ns;
};

// Shared-memory descriptor of a scale atom for tcgen05.cp: no swizzle, 8-row core matrices
// of 16-byte rows stored contiguously (stride 128 bytes between 8-row groups).
__device__ __forceinline__ uint64_t desc_atom(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(512u >> 4) << 16;
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// 32 lanes x 128 bits of shared memory to TMEM, repeated into all four lane quarters.
__device__ __forceinline__ void tmem_cp_atom(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

// Instruction descriptor of kind::mxf8f6f4: e4m3 x e4m3, fp32 accumulate, K-major A and B,
// UE8M0 scales (bit 23), B scale-factor id at bits 4-5, A scale-factor id at bits 29-30.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB0x,
                      const __grid_constant__ CUtensorMap tmB1x, const __grid_constant__ CUtensorMap tmSA,
                      const __grid_constant__ CUtensorMap tmSB0, const __grid_constant__ CUtensorMap tmSB1,
                      const __grid_constant__ CUtensorMap tmSB0x, const __grid_constant__ CUtensorMap tmSB1x,
                      const MxParams p) {
  using S = MxSmem;
  constexpr int kStages = S::kStages, kBBytes = S::kBBytes, kStageBytes = S::kStageBytes;
  constexpr int TM = BM;  // rows of an m tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sSF = sB + kStages * kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* mt_prefix = reinterpret_cast<int32_t*>(bars + 32);
  int32_t* seg_rows = mt_prefix + kMaxGroups;
  uint8_t* sEpi = reinterpret_cast<uint8_t*>(seg_rows + kMaxGroups);  // [kEpiWarps][32 rows][64 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = p.G + p.has_extra;
  const int kblocks = p.K / BK;
  const int unit = blockIdx.x, nunits = gridDim.x;  // persistent tile walkers

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);  // one arrival per epilogue warp
    mbar_init(drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmSA);
  }
  if (warp == 1) tmem_alloc_cg<1>(tmem_slot, kTmemCols);
  if (warp == 2) build_tile_prefix(p.offsets, p.G, ngroups, p.T_extra, TM, lane, seg_rows, mt_prefix);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.n_tiles * mt_prefix[ngroups];

  if (warp == 0) {
    // ======================= TMA producer (A rows, B rows and the stage's scale atoms)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
        const bool extra = c.g >= p.G;
        const int64_t gofs = extra ? (int64_t)p.a2_row_base : (int64_t)p.offsets[c.g];
        const int a_row = (int)gofs + c.mb * TM;
        const int a_atom = (int)(mx_group_atom_base(gofs, c.g) + c.mb);
        const CUtensorMap* tb0 = extra ? &tmB0x : &tmB0;
        const CUtensorMap* tb1 = extra ? &tmB1x : &tmB1;
        const CUtensorMap* ts0 = extra ? &tmSB0x : &tmSB0;
        const CUtensorMap* ts1 = extra ? &tmSB1x : &tmSB1;
        const int b_tile_rows = EPI == MX_SWIGLU_Q8 ? BN / 2 : BN;
        const int b_row = (extra ? 0 : c.g * p.b_group_rows) + c.nb * b_tile_rows;
        const int b_atom = b_row / 128;  // b_row is a multiple of 128
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * kBBytes;
          uint8_t* sf_dst = sSF + stage * kSfBytes;
          const int sa_y = a_atom * kblocks + kb;
          const int sb0_y = (EPI == MX_SWIGLU_Q8 ? b_atom : b_atom) * kblocks + kb;
          const int sb1_y = (EPI == MX_SWIGLU_Q8 ? b_atom : b_atom + 1) * kblocks + kb;
          const CUtensorMap* tsb1 = EPI == MX_SWIGLU_Q8 ? ts1 : ts0;
          mbar_arrive_expect_tx(&full[stage], kStageBytes);
          tma_load_2d(&tmA, a_dst, &full[stage], kb * BK, a_row);
          if (EPI == MX_SWIGLU_Q8) {
            tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);
            tma_load_2d(tb1, b_dst + (BN / 2) * BK, &full[stage], kb * BK, b_row);
          } else {
            tma_load_2d(tb0, b_dst, &full[stage], kb * BK, b_row);
          }
          tma_load_2d(&tmSA, sf_dst, &full[stage], 0, sa_y);
          tma_load_2d(ts0, sf_dst + kAtomBytes, &full[stage], 0, sb0_y);
          tma_load_2d(tsb1, sf_dst + 2 * kAtomBytes, &full[stage], 0, sb1_y);
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      // wind down: every issued load has landed and been consumed before the block exits
      const int used = issued < kStages ? (int)issued : kStages;
      for (int i = 0; i < used; ++i) {
        const int s = (stage - 1 - i + 2 * kStages) % kStages;
        const uint32_t ph = (stage - 1 - i < 0) ? (phase ^ 1) : phase;
        if (ok) ok = mbar_wait(&empty[s], ph, abort, p.timeout_ns, p.status);
        if (!ok) mbar_wait_drain(&full[s], ph, p.timeout_ns, p.status);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
        // the epilogue has taken the previous tile's accumulator out of TMEM
        if (!mbar_wait(acc_empty, acc_phase ^ 1, abort, p.timeout_ns, p.status)) { ok = false; break; }
        acc_phase ^= 1;
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort, p.timeout_ns, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kBBytes);
          const uint32_t sf_addr = smem_addr(sSF + stage * kSfBytes);
          const uint32_t sfa_t = tmem_base + kSfCol0 + stage * kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4;
          tmem_cp_atom(sfa_t, desc_atom(sf_addr));
          tmem_cp_atom(sfb_t, desc_atom(sf_addr + kAtomBytes));
          tmem_cp_atom(sfb_t + 4, desc_atom(sf_addr + 2 * kAtomBytes));
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)  // K = 32 e4m3 per instruction: +32 bytes, scale id k
            mma_mx(tmem_base, desc_k_sw128(a_addr + k * 32), desc_k_sw128(b_addr + k * 32),
                   idesc_mx(TM, BN, (uint32_t)k), sfa_t, sfb_t, (kb | k) != 0);
          mma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit(acc_full);
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0, p.timeout_ns, p.status);
    }
  } else {
    // ======================= epilogue: warps 2..9
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;  // which 128 of the tile's 256 columns this warp owns
    const int r = quarter * 32 + lane;  // TMEM lane = row of the tile
    uint8_t* stage = sEpi + ew * kEpiStageBytes;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = unit; tile < total_tiles && ok; tile += nunits) {
      const TileCoord c = decode_tile(tile, mt_prefix, ngroups, p.n_tiles, seg_rows, TM);
      const bool extra = c.g >= p.G;
      ok = mbar_wait(acc_full, acc_phase, abort, p.timeout_ns, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      acc_phase ^= 1;
      tc_fence_after();
      const uint32_t t = tmem_base + ((uint32_t)(quarter * 32) << 16);
      uint32_t v[128];
      if (EPI == MX_SWIGLU_Q8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tmem_ld16(t + half * 64 + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * q]));
          tmem_ld16(t + 128 + half * 64 + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&v[64 + 16 * q]));
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) tmem_ld16(t + half * 128 + 16 * q, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * q]));
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();  // every lane's loads are complete: one arrival per warp
      if (lane == 0) mbar_arrive_relaxed(acc_empty);

      const int64_t gofs = extra ? (int64_t)p.a2_row_base : (int64_t)p.offsets[c.g];
      const int64_t row0 = (extra ? p.out_extra_base : gofs) + c.mb * TM + quarter * 32;
      const int live_rows = c.rows - quarter * 32;  // rows of this warp inside the segment
      if (EPI == MX_SWIGLU_Q8) {
        // 64 bytes of h codes per thread per tile: direct 16-byte stores
        if (r < c.rows) {
          uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + (row0 + lane) * p.ldc + c.nb * 128 + half * 64;
          uint32_t codes = 0;
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            float h[32];
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(v[32 * blk + i]);
              h[i] = g / (1.0f + __expf(-g)) * __uint_as_float(v[64 + 32 * blk + i]);
              amax = fmaxf(amax, fabsf(h[i]));
            }
            const int s = mx_scale_exp(amax);
            const float inv = mx_inv_scale(s);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = e4m3x4(__fmul_rn(h[4 * i], inv), __fmul_rn(h[4 * i + 1], inv), __fmul_rn(h[4 * i + 2], inv),
                            __fmul_rn(h[4 * i + 3], inv));
            reinterpret_cast<uint4*>(out + 32 * blk)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(out + 32 * blk)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            codes |= (uint32_t)(s + 127) << (8 * blk);
          }
          // blocks 2*half and 2*half + 1 of the h stage nb, in the tile's atom row
          const int64_t atom = mx_group_atom_base(gofs, c.g) + c.mb;
          *reinterpret_cast<uint16_t*>(p.out_sf + mx_atom_byte(atom, c.nb, p.ldc / 128, r) + 2 * half) =
              (uint16_t)codes;
        }
      } else {
        // 256 bytes of bf16 per thread per tile: staged through shared memory, 32 columns
        // at a time, so that the stores are coalesced
        uint8_t* out = reinterpret_cast<uint8_t*>(p.out) + (row0 * p.ldc + c.nb * BN + half * 128) * 2;
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 32 columns (64 bytes of bf16) per pass
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t w4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int i = 32 * q + 8 * c4 + 2 * j;
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
              w4[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            stage_piece(stage, lane, c4, make_uint4(w4[0], w4[1], w4[2], w4[3]));
          }
          flush_rows_64B(stage, lane, out + 64 * q, (int64_t)p.ldc * 2, live_rows);
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

// Scale atoms as rows of 128 uint32 (one 512-byte box per atom, no swizzle).
bool make_atoms(CUtensorMap* m, const void* base, uint64_t atoms) {
  return make_tmap_linear(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, atoms, 128, 1, 128);
}

struct MxMaps {
  CUtensorMap a, b0, b1, b0x, b1x, sa, sb0, sb1, sb0x, sb1x;
};

template <int EPI>
cudaError_t launch(const MxMaps& m, const MxParams& p, int64_t max_tiles, cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  auto kern = tc_gemm_mx_kernel<EPI>;
  const size_t smem = MxSmem::kBytes;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = (int)std::min<int64_t>(num_sms(), max_tiles);
  kern<<<grid, kThreads, smem, s>>>(m.a, m.b0, m.b1, m.b0x, m.b1x, m.sa, m.sb0, m.sb1, m.sb0x, m.sb1x, p);
  return cudaGetLastError();
}

}  // namespace

bool mx_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.xfer_dtype == MOE_DTYPE_MXE4M3 && c.H % 256 == 0 && c.F % 128 == 0 &&
         c.E + 1 <= kMaxGroups;
}

cudaError_t launch_grouped_mlp_mx(const moe_config_t& c, const void* xd, const void* xd_sf, const int32_t* offsets,
                                  const moe_weights_t& w, void* h, void* h_sf, void* yd, DeviceStatus* st,
                                  cudaStream_t s) {
  const int64_t R = routed_rows(c), rows = total_rows(c);
  const bool shared = c.n_shared != 0;
  // Single-CTA tiles: a CTA-pair form of this kernel computed the same results but ran
  // slower (10.67 against 9.76 ms on the DeepSeek-V3-shaped MXFP8 layer): its accumulator
  // has to stay single-buffered (two 256-column accumulators and the scale factors exceed
  // 512 TMEM columns), so every tile boundary waits for both CTAs' epilogues, and 256-row
  // tiles double the padding of ragged segment tails.
  const int64_t atoms_act = mx_act_atom_rows(c);
  // ---- GEMM1: h = mx(silu(A Wg^T) * (A Wu^T)); the shared expert's A = dispatched rows R..
  MxMaps m{};
  bool ok = make_u8(&m.a, xd, rows, c.H, BM) && make_u8(&m.b0, w.w_gate, (uint64_t)c.E * c.F, c.H, 128) &&
            make_u8(&m.b1, w.w_up, (uint64_t)c.E * c.F, c.H, 128) &&
            make_atoms(&m.sa, xd_sf, (uint64_t)atoms_act * (c.H / 128)) &&
            make_atoms(&m.sb0, w.s_gate, (uint64_t)c.E * c.F / 128 * (c.H / 128)) &&
            make_atoms(&m.sb1, w.s_up, (uint64_t)c.E * c.F / 128 * (c.H / 128));
  if (shared)
    ok = ok && make_u8(&m.b0x, w.ws_gate, c.F, c.H, 128) && make_u8(&m.b1x, w.ws_up, c.F, c.H, 128) &&
         make_atoms(&m.sb0x, w.ss_gate, (uint64_t)c.F / 128 * (c.H / 128)) &&
         make_atoms(&m.sb1x, w.ss_up, (uint64_t)c.F / 128 * (c.H / 128));
  else { m.b0x = m.b0; m.b1x = m.b1; m.sb0x = m.sb0; m.sb1x = m.sb1; }
  if (!ok) return cudaErrorInvalidValue;
  MxParams p{};
  p.offsets = offsets;
  p.G = c.E;
  p.has_extra = shared ? 1 : 0;
  p.T_extra = c.T;
  p.a2_row_base = (int)R;
  p.out_extra_base = R;
  p.K = c.H;
  p.n_tiles = c.F / 128;
  p.b_group_rows = c.F;
  p.ldc = c.F;
  p.out = h;
  p.out_sf = static_cast<uint8_t*>(h_sf);
  p.status = st;
  p.timeout_ns = kTimeoutNs;
  const int64_t mt_bound = ceil_div(R, BM) + c.E + (shared ? ceil_div(c.T, BM) : 0);
  cudaError_t e = launch<MX_SWIGLU_Q8>(m, p, mt_bound * p.n_tiles, s);
  if (e != cudaSuccess) return e;
  // ---- GEMM2: yd = h Wd^T with both operands' MX scales, bf16 out
  MxMaps m2{};
  ok = make_u8(&m2.a, h, rows, c.F, BM) && make_u8(&m2.b0, w.w_down, (uint64_t)c.E * c.H, c.F, BN) &&
       make_atoms(&m2.sa, h_sf, (uint64_t)atoms_act * (c.F / 128)) &&
       make_atoms(&m2.sb0, w.s_down, (uint64_t)c.E * c.H / 128 * (c.F / 128));
  if (shared)
    ok = ok && make_u8(&m2.b0x, w.ws_down, c.H, c.F, BN) &&
         make_atoms(&m2.sb0x, w.ss_down, (uint64_t)c.H / 128 * (c.F / 128));
  else { m2.b0x = m2.b0; m2.sb0x = m2.sb0; }
  if (!ok) return cudaErrorInvalidValue;
  m2.b1 = m2.b0; m2.b1x = m2.b0x; m2.sb1 = m2.sb0; m2.sb1x = m2.sb0x;
  p.K = c.F;
  p.n_tiles = c.H / BN;
  p.b_group_rows = c.H;
  p.ldc = c.H;
  p.out = yd;
  p.out_sf = nullptr;
  return launch<MX_STORE_BF16>(m2, p, mt_bound * p.n_tiles, s);
}

}  // namespace tc
}  // namespace moe
