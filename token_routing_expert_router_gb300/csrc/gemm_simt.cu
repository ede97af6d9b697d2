// SIMT grouped GEMM with fp32 FFMA accumulation: C[r, n] = sum_k A[r, k] * B[n, k] per
// group. It is the exact-fp32 path of the expert MLP (TF32 tensor cores cannot hold a
// 1e-5 relative error) and of the router logits for small expert counts. The grouped form
// reads the per-expert row ranges from device memory ("Scalable Training of Mixture-of-
// Experts Models with Megatron Core" summary, section 2.4: grouped GEMM, device-initiated
// kernels); every block finds its (group, row tile) itself, so no host sync is needed.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <bool BF16>
__device__ __forceinline__ float ld_elem(const void* p, int64_t i) {
  if (BF16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(p)[i] << 16);
  return reinterpret_cast<const float*>(p)[i];
}

template <bool BF16>
__device__ __forceinline__ void st_elem(void* p, int64_t i, float v) {
  if (BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else reinterpret_cast<float*>(p)[i] = v;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

template <bool BF16, int MODE>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(SimtGemmArgs a) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[2][BK][BN + 4];

  // ---- which group and row tile this block computes
  int mt = blockIdx.y;
  int g = 0, M = 0;
  int64_t row_in = 0, row_out = 0;
  const void* A = a.A;
  const void* B0 = a.B0;
  const void* B1 = a.B1;
  const int K = a.K, N = a.N;
  if (a.M_static >= 0) {
    M = a.M_static;
    if (mt >= (int)ceil_div(M, BM)) return;
  } else {
    const int G = a.G + a.extra_group;
    for (g = 0; g < G; ++g) {
      M = (g < a.G) ? a.offsets[g + 1] - a.offsets[g] : a.T_extra;
      const int tiles = (int)ceil_div(M, BM);
      if (mt < tiles) break;
      mt -= tiles;
    }
    if (g == G) return;
    if (g < a.G) {
      row_in = a.offsets[g];
      row_out = row_in;
      B0 = (const char*)a.B0 + (int64_t)g * N * K * (BF16 ? 2 : 4);
      if (MODE == 1) B1 = (const char*)a.B1 + (int64_t)g * N * K * (BF16 ? 2 : 4);
    } else {
      A = a.A_extra;
      row_in = 0;
      row_out = a.routed_rows;
      B0 = a.B0_extra;
      B1 = a.B1_extra;
    }
  }
  const int m0 = mt * BM, n0 = blockIdx.x * BN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;

  float acc0[4][4], acc1[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc0[i][j] = 0.0f; acc1[i][j] = 0.0f; }

  // 64 x 16 tiles: each thread loads 4 elements of A and 4 of each B, the next K tile's
  // into registers while the current one is multiplied
  float ra[4], rb0[4], rb1[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int e = threadIdx.x + l * NT;  // 0..1023
      const int r = e / BK, kk = e % BK;
      const int gr = m0 + r, gk = k0 + kk, gn = n0 + r;
      ra[l] = (gr < M && gk < K) ? ld_elem<BF16>(A, (row_in + gr) * K + gk) : 0.0f;
      rb0[l] = (gn < N && gk < K) ? ld_elem<BF16>(B0, (int64_t)gn * K + gk) : 0.0f;
      if (MODE == 1) rb1[l] = (gn < N && gk < K) ? ld_elem<BF16>(B1, (int64_t)gn * K + gk) : 0.0f;
    }
  };
  if (K > 0) load(0);
  for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int e = threadIdx.x + l * NT;
      const int r = e / BK, kk = e % BK;
      As[kk][r] = ra[l];
      Bs[0][kk][r] = rb0[l];
      if (MODE == 1) Bs[1][kk][r] = rb1[l];
    }
    __syncthreads();
    if (k0 + BK < K) load(k0 + BK);
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4], cv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { av[i] = As[kk][ty * 4 + i]; bv[i] = Bs[0][kk][tx * 4 + i]; }
      if (MODE == 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) cv[i] = Bs[1][kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc0[i][j] = __fmaf_rn(av[i], bv[j], acc0[i][j]);
          if (MODE == 1) acc1[i][j] = __fmaf_rn(av[i], cv[j], acc1[i][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = m0 + ty * 4 + i;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      const int64_t o = (row_out + r) * N + n;
      if (MODE == 0) {
        float v = acc0[i][j];
        if (a.bias) v += a.bias[n];
        reinterpret_cast<float*>(a.C)[o] = v;
      } else if (MODE == 1) {
        st_elem<BF16>(a.C, o, silu_mul(acc0[i][j], acc1[i][j]));
      } else {
        st_elem<BF16>(a.C, o, acc0[i][j]);
      }
    }
  }
}

// ---------------------------------------------------------------- small fp32 problems
// With a few hundred rows (the tiny layer: 512 routed rows, K = 128 or 256) the 64 x 64
// kernel above runs 32-64 blocks that each wait on memory once per 16-deep K step. Here a
// block computes a 32 x 32 tile and copies the whole K extent of its 32 A rows and 32 B rows
// (two B tiles for the gate/up mode) into shared memory at once, so it waits on memory once
// and the grid has four times as many blocks. Each output is still summed in ascending k
// with one FMA per product, as above, so both kernels give the same bits.
constexpr int SBM = 32, SBN = 32, SNT = 128, kSmallMaxK = 256;

__device__ __forceinline__ void cp_async16_f(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(SNT) simt_small_kernel(SimtGemmArgs a) {
  extern __shared__ float4 s_small[];
  const int K = a.K, N = a.N, ld = K + 4;  // row pitch: 16-byte rows, ld = 4 (mod 32) banks for K % 32 == 0
  float* As = reinterpret_cast<float*>(s_small);
  float* Bs0 = As + SBM * ld;
  float* Bs1 = Bs0 + SBN * ld;  // MODE 1: the up rows

  int mt = blockIdx.y;
  int M = 0;
  int64_t row_in = 0, row_out = 0;
  const float* A = static_cast<const float*>(a.A);
  const float* B0 = static_cast<const float*>(a.B0);
  const float* B1 = static_cast<const float*>(a.B1);
  if (a.M_static >= 0) {
    M = a.M_static;
    if (mt >= (int)ceil_div(M, SBM)) return;
  } else {
    const int G = a.G + a.extra_group;
    int g = 0;
    for (; g < G; ++g) {
      M = (g < a.G) ? a.offsets[g + 1] - a.offsets[g] : a.T_extra;
      const int tiles = (int)ceil_div(M, SBM);
      if (mt < tiles) break;
      mt -= tiles;
    }
    if (g == G) return;
    if (g < a.G) {
      row_in = a.offsets[g];
      row_out = row_in;
      B0 += (int64_t)g * N * K;
      if (MODE == 1) B1 += (int64_t)g * N * K;
    } else {
      A = static_cast<const float*>(a.A_extra);
      row_out = a.routed_rows;
      B0 = static_cast<const float*>(a.B0_extra);
      B1 = static_cast<const float*>(a.B1_extra);
    }
  }
  const int m0 = mt * SBM, n0 = blockIdx.x * SBN;

  // ---- the whole K extent into shared memory (rows past the tile's end read as zeros)
  const int kv = K / 4;
  for (int i = threadIdx.x; i < SBM * kv; i += SNT) {
    const int r = i / kv, c = 4 * (i - (i / kv) * kv);
    float* da = As + r * ld + c;
    if (m0 + r < M) cp_async16_f(da, A + (row_in + m0 + r) * K + c);
    else *reinterpret_cast<float4*>(da) = make_float4(0.f, 0.f, 0.f, 0.f);
    float* db = Bs0 + r * ld + c;
    if (n0 + r < N) cp_async16_f(db, B0 + (int64_t)(n0 + r) * K + c);
    else *reinterpret_cast<float4*>(db) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (MODE == 1) {
      float* du = Bs1 + r * ld + c;
      if (n0 + r < N) cp_async16_f(du, B1 + (int64_t)(n0 + r) * K + c);
      else *reinterpret_cast<float4*>(du) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // ---- thread (tx, ty): rows ty + 16 i (i < 2), columns tx + 8 j (j < 4); four k a step
  const int tx = threadIdx.x & 7, ty = threadIdx.x >> 3;
  float acc0[2][4], acc1[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { acc0[i][j] = 0.0f; acc1[i][j] = 0.0f; }
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 av[2], bv[4], cv[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) av[i] = *reinterpret_cast<const float4*>(As + (ty + 16 * i) * ld + k);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bv[j] = *reinterpret_cast<const float4*>(Bs0 + (tx + 8 * j) * ld + k);
      if (MODE == 1) cv[j] = *reinterpret_cast<const float4*>(Bs1 + (tx + 8 * j) * ld + k);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc0[i][j] = __fmaf_rn(av[i].x, bv[j].x, acc0[i][j]);
        acc0[i][j] = __fmaf_rn(av[i].y, bv[j].y, acc0[i][j]);
        acc0[i][j] = __fmaf_rn(av[i].z, bv[j].z, acc0[i][j]);
        acc0[i][j] = __fmaf_rn(av[i].w, bv[j].w, acc0[i][j]);
        if (MODE == 1) {
          acc1[i][j] = __fmaf_rn(av[i].x, cv[j].x, acc1[i][j]);
          acc1[i][j] = __fmaf_rn(av[i].y, cv[j].y, acc1[i][j]);
          acc1[i][j] = __fmaf_rn(av[i].z, cv[j].z, acc1[i][j]);
          acc1[i][j] = __fmaf_rn(av[i].w, cv[j].w, acc1[i][j]);
        }
      }
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = m0 + ty + 16 * i;
    if (r >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 8 * j;
      if (n >= N) continue;
      const int64_t o = (row_out + r) * N + n;
      float* C = static_cast<float*>(a.C);
      if (MODE == 0) C[o] = a.bias ? acc0[i][j] + a.bias[n] : acc0[i][j];
      else if (MODE == 1) C[o] = silu_mul(acc0[i][j], acc1[i][j]);
      else C[o] = acc0[i][j];
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// fp32, K a multiple of 4 up to kSmallMaxK, 16-byte aligned operands, and a problem the
// 64 x 64 grid would cover with fewer blocks than two per SM.
bool small_form(const SimtGemmArgs& a, int64_t mtiles64, int sms) {
  if (a.act_bf16 || a.K <= 0 || a.K % 4 != 0 || a.K > kSmallMaxK) return false;
  if (ceil_div(a.N, BN) * mtiles64 >= 2LL * sms) return false;
  const void* ptrs[] = {a.A, a.A_extra, a.B0, a.B1, a.B0_extra, a.B1_extra};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return false;
  return true;
}

template <int MODE>
cudaError_t launch_small(const SimtGemmArgs& a, int64_t mtiles, cudaStream_t s) {
  const size_t smem = (size_t)(MODE == 1 ? 3 : 2) * SBM * (a.K + 4) * sizeof(float);
  static bool attr_set = false;  // per instantiation: room for K = kSmallMaxK
  if (!attr_set) {
    const int max_smem = (MODE == 1 ? 3 : 2) * SBM * (kSmallMaxK + 4) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(simt_small_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         max_smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const dim3 grid((unsigned)ceil_div(a.N, SBN), (unsigned)mtiles);
  simt_small_kernel<MODE><<<grid, SNT, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemmArgs& a, cudaStream_t s) {
  int64_t mtiles;
  if (a.M_static >= 0) {
    mtiles = ceil_div(a.M_static, BM);
  } else {
    // upper bound over any split of R rows into G groups (+ the extra group)
    mtiles = ceil_div(a.routed_rows, BM) + a.G + (a.extra_group ? ceil_div(a.T_extra, BM) : 0);
  }
  if (mtiles == 0 || a.N == 0) return cudaSuccess;
  if (mtiles > 65535) return cudaErrorInvalidValue;
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  if (small_form(a, mtiles, sms)) {
    // the same bound at 32-row tiles
    const int64_t mt32 = a.M_static >= 0 ? ceil_div(a.M_static, SBM)
                                         : ceil_div(a.routed_rows, SBM) + a.G +
                                               (a.extra_group ? ceil_div(a.T_extra, SBM) : 0);
    if (mt32 <= 65535) {
      if (a.mode == 0) return launch_small<0>(a, mt32, s);
      if (a.mode == 1) return launch_small<1>(a, mt32, s);
      return launch_small<2>(a, mt32, s);
    }
  }
  const dim3 grid((unsigned)ceil_div(a.N, BN), (unsigned)mtiles);
#define MOE_SIMT(BF, MODE) simt_gemm_kernel<BF, MODE><<<grid, NT, 0, s>>>(a)
  if (a.act_bf16) {
    if (a.mode == 0) MOE_SIMT(true, 0);
    else if (a.mode == 1) MOE_SIMT(true, 1);
    else MOE_SIMT(true, 2);
  } else {
    if (a.mode == 0) MOE_SIMT(false, 0);
    else if (a.mode == 1) MOE_SIMT(false, 1);
    else MOE_SIMT(false, 2);
  }
#undef MOE_SIMT
  return cudaGetLastError();
}

}  // namespace moe
