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
