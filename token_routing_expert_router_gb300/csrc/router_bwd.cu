// The router's backward: the gradient of the layer's output (and of the auxiliary
// load-balancing loss) with respect to the router logits, the router weight and bias, and
// the input's share through the router. The router is the linear map that scores every
// token against the experts ("Scalable Training of Mixture-of-Experts Models with
// Megatron Core" summary, "O essencial"); the routing weights are the softmax or sigmoid
// of those scores over the chosen experts, so with the choice held fixed the chain rule
// runs through the weight step and then through the linear map.
//
//  1. logit_grad_kernel: one warp per token, fp32. dL/dw (the combine backward's
//     routing-weight gradient) through the weight step, plus the auxiliary loss's gradient
//     through the normalised probabilities of all experts.
//  2. wgrad_kernel: dW_router = dl^T x and the bias gradient (column sums of dl), as a
//     register-tiled fp32 SIMT product split over token slices; the slices' partial sums
//     are added in slice order by sum_slices_kernel, so results do not depend on timing.
//  3. input_grad_kernel: dx[t] = sum_e dl[t,e] W_router[e] + sum_j dxd[tok_row[t,j]]
//     (+ dxd[R + t]): the router's share and the dispatch backward's gather-reduce in one
//     pass over dx, accumulated in fp32 and rounded to bf16 once.
// With many experts (E a multiple of 128, H of 256, bf16) the two products are dense enough for
// the tensor cores: dl is also written in bf16, dW_router = dl^T x and dx_r = dl W_router
// run as the expert backward's tcgen05 GEMMs over the tokens as one group, the bias
// gradient is a column sum of dl, and dx = dx_r + the dispatch rows is the combine kernel
// with one extra row.
#include <algorithm>

#include "gemm_tc.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// ---------------------------------------------------------------------------------------
// 1. Logit gradient. Lane e % 32 owns experts e = lane + 32 i (i < EPL); lane j < k owns
// the token's j-th choice. The row is staged in shared memory so the chosen experts' terms
// (one lane each, distinct experts) land on the owning slots before one coalesced store.
// ---------------------------------------------------------------------------------------
constexpr int kLgWarps = 8;
constexpr int kMaxE = 512;

template <int EPL>
__global__ void __launch_bounds__(kLgWarps * 32)
    logit_grad_kernel(const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                      const float* __restrict__ dtopk_w, int T, int E, int k, int score_fn, int renorm, float rho,
                      const int32_t* __restrict__ counts, float aux_a0, float* __restrict__ dl,
                      __nv_bfloat16* __restrict__ dlb, int32_t* __restrict__ slice_offsets, int slice, int slices,
                      DeviceStatus* st) {
  __shared__ float row_s[kLgWarps][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the token slices of the tensor-core weight gradient (read by a later launch)
  if (slice_offsets != nullptr && blockIdx.x == 0 && (int)threadIdx.x <= slices)
    slice_offsets[threadIdx.x] = (int)min((int64_t)threadIdx.x * slice, (int64_t)T);
  const int t = blockIdx.x * kLgWarps + warp;
  if (t >= T) return;
  const float* l = logits + (int64_t)t * E;
  float lv[EPL], d[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    lv[i] = e < E ? l[e] : -INFINITY;
    d[i] = 0.0f;
  }
  // this lane's choice
  int ij = 0;
  float gj = 0.0f, lj = -INFINITY;
  bool bad = false;
  if (lane < k) {
    ij = topk_idx[(int64_t)t * k + lane];
    bad = ij < 0 || ij >= E;
    if (bad) ij = 0;
    gj = rho * dtopk_w[(int64_t)t * k + lane];
    lj = l[ij];
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);
    return;
  }
  const bool need_softmax_all = score_fn == 0 && (!renorm || counts != nullptr);
  float m_all = 0.0f, inv_den_all = 0.0f;
  if (need_softmax_all) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, lv[i]);
    m_all = warp_max(m);
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) s += lane + 32 * i < E ? expf(lv[i] - m_all) : 0.0f;
    inv_den_all = 1.0f / warp_sum(s);
  }
  float dj = 0.0f;  // the chosen expert's own term, added at slot ij
  if (score_fn == 0) {
    if (!renorm) {
      // p = softmax over all experts: dl_e = [e chosen] g p_e - p_e sum_j g_j p_j
      const float pj = lane < k ? expf(lj - m_all) * inv_den_all : 0.0f;
      const float c = warp_sum(gj * pj);
#pragma unroll
      for (int i = 0; i < EPL; ++i) d[i] = -(expf(lv[i] - m_all) * inv_den_all) * c;
      dj = gj * pj;
    } else {
      // q = softmax over the chosen: dl_j = q_j (g_j - sum_i g_i q_i)
      const float mk = warp_max(lj);
      const float vj = lane < k ? expf(lj - mk) : 0.0f;
      const float qj = vj / warp_sum(vj);
      const float c = warp_sum(gj * qj);
      dj = qj * (gj - c);
    }
  } else {
    const float sj = lane < k ? 1.0f / (1.0f + expf(-lj)) : 0.0f;
    if (renorm) {
      // w~ = s / S over the chosen: dl_j = s_j (1 - s_j) (g_j - sum_i g_i w~_i) / S
      const float S = warp_sum(sj);
      const float c = warp_sum(gj * sj) / S;
      dj = sj * (1.0f - sj) * (gj - c) / S;
    } else {
      dj = gj * sj * (1.0f - sj);
    }
  }
  if (counts != nullptr) {
    // auxiliary loss: dL/dp_hat[t,e] = a_e = aux_a0 * c_e for every token, p_hat the
    // softmax over all experts or the sigmoids divided by their sum
    float ph[EPL], sv[EPL], a[EPL], inv = 1.0f, csum = 0.0f;
    if (score_fn == 0) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) ph[i] = expf(lv[i] - m_all) * inv_den_all;  // 0 past E
    } else {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        sv[i] = lane + 32 * i < E ? 1.0f / (1.0f + expf(-lv[i])) : 0.0f;
        s += sv[i];
      }
      inv = 1.0f / warp_sum(s);
#pragma unroll
      for (int i = 0; i < EPL; ++i) ph[i] = sv[i] * inv;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      a[i] = e < E ? aux_a0 * (float)counts[e] : 0.0f;
      csum += a[i] * ph[i];
    }
    const float c = warp_sum(csum);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      d[i] += score_fn == 0 ? ph[i] * (a[i] - c) : sv[i] * (1.0f - sv[i]) * (a[i] - c) * inv;
  }
  float* row = row_s[warp];
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) row[lane + 32 * i] = d[i];
  __syncwarp();
  if (lane < k) row[ij] += dj;
  __syncwarp();
  float* out = dl + (int64_t)t * E;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) out[lane + 32 * i] = row[lane + 32 * i];
  if (dlb != nullptr) {
    __nv_bfloat16* ob = dlb + (int64_t)t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) ob[lane + 32 * i] = __float2bfloat16_rn(row[lane + 32 * i]);
  }
}

// Column sums of src [rows, cols] over row slice b (rows [b * slice, + slice)) -> out[b, :]:
// the bias gradient's two levels (dl's token slices, then the slices' partials). With
// cols <= 256 the block's threads split into 256 / cols row phases; every thread keeps four
// independent partial sums (rows i = 0, 1, 2, 3 mod 4 of its phase) so that loads overlap,
// and the partials and then the phases are added in a fixed order.
__global__ void __launch_bounds__(256) colsum_kernel(const float* __restrict__ src, int rows, int cols, int slice,
                                                     float* __restrict__ out) {
  __shared__ float red[256];
  const int r0 = blockIdx.x * slice, r1 = min(rows, r0 + slice);
  const int nph = cols <= 256 ? 256 / cols : 1;
  for (int cbase = 0; cbase < cols; cbase += 256) {
    const int c = cbase + (cols <= 256 ? (int)threadIdx.x % cols : (int)threadIdx.x);
    const int ph = cols <= 256 ? (int)threadIdx.x / cols : 0;
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (ph < nph && c < cols) {
      int i = 0;
      for (int r = r0 + ph; r < r1; r += nph, ++i) a[i & 3] += src[(int64_t)r * cols + c];
    }
    __syncthreads();
    red[threadIdx.x] = (a[0] + a[1]) + (a[2] + a[3]);
    __syncthreads();
    if (ph == 0 && c < cols) {
      float v = red[threadIdx.x];
      for (int q = 1; q < nph; ++q) v += red[threadIdx.x + q * cols];
      out[(int64_t)blockIdx.x * cols + c] = v;
    }
  }
}

__global__ void __launch_bounds__(256) to_bf16_kernel(const float* __restrict__ src, int64_t n,
                                                      __nv_bfloat16* __restrict__ dst) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

// ---------------------------------------------------------------------------------------
// 2. dW_router[e, h] = sum_t dl[t, e] x[t, h] over token slice z, and the bias partial
// sum_t dl[t, e]. Block tile BM experts x 128 columns; thread (ty, tx) of 8 x 32 holds
// BM/8 experts x 4 columns; 32 tokens per shared-memory stage, the next stage's global
// loads issued before the current stage's products.
// ---------------------------------------------------------------------------------------
constexpr int kWgBN = 128, kWgBK = 32, kWgThreads = 256;
constexpr int kBiasSlice = 128;  // tokens per slice of the tensor-core path's bias gradient

template <int BM, bool BF16>
__global__ void __launch_bounds__(kWgThreads)
    wgrad_kernel(const float* __restrict__ dl, const void* __restrict__ x_, int T, int E, int H, int slice,
                 float* __restrict__ out, float* __restrict__ bias_out) {
  constexpr int TM = BM / 8;
  constexpr int AL = BM * kWgBK / kWgThreads;           // dl elements per thread per stage
  constexpr int VE = BF16 ? 8 : 4;                       // x elements per 16-byte vector
  constexpr int BV = kWgBK * kWgBN / VE / kWgThreads;    // x vectors per thread per stage
  __shared__ __align__(16) float As[kWgBK][BM];
  __shared__ __align__(16) float Bs[kWgBK][kWgBN];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int h0 = blockIdx.x * kWgBN, e0 = blockIdx.y * BM;
  const int t_begin = blockIdx.z * slice, t_end = min(T, t_begin + slice);
  const bool do_bias = bias_out != nullptr && blockIdx.x == 0;

  float acc[TM][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  float bacc = 0.0f;

  float ra[AL];
  uint4 rb[BV];
  auto load = [&](int t0) {
#pragma unroll
    for (int q = 0; q < AL; ++q) {
      const int idx = tid + q * kWgThreads, kk = idx / BM, m = idx % BM;
      const int t = t0 + kk, e = e0 + m;
      ra[q] = (t < t_end && e < E) ? dl[(int64_t)t * E + e] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < BV; ++q) {
      const int v = tid + q * kWgThreads, kk = v / (kWgBN / VE), n = (v % (kWgBN / VE)) * VE;
      const int t = t0 + kk, h = h0 + n;
      rb[q] = (t < t_end && h < H)
                  ? __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(x_) +
                                                         ((int64_t)t * H + h) * (BF16 ? 2 : 4)))
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int q = 0; q < AL; ++q) {
      const int idx = tid + q * kWgThreads;
      As[idx / BM][idx % BM] = ra[q];
    }
#pragma unroll
    for (int q = 0; q < BV; ++q) {
      const int v = tid + q * kWgThreads, kk = v / (kWgBN / VE), n = (v % (kWgBN / VE)) * VE;
      if (BF16) {
        const float4 lo = make_float4(bf16_lo(rb[q].x), bf16_hi(rb[q].x), bf16_lo(rb[q].y), bf16_hi(rb[q].y));
        const float4 hi = make_float4(bf16_lo(rb[q].z), bf16_hi(rb[q].z), bf16_lo(rb[q].w), bf16_hi(rb[q].w));
        *reinterpret_cast<float4*>(&Bs[kk][n]) = lo;
        *reinterpret_cast<float4*>(&Bs[kk][n + 4]) = hi;
      } else {
        *reinterpret_cast<float4*>(&Bs[kk][n]) = make_float4(__uint_as_float(rb[q].x), __uint_as_float(rb[q].y),
                                                             __uint_as_float(rb[q].z), __uint_as_float(rb[q].w));
      }
    }
  };

  if (t_begin < t_end) load(t_begin);
  for (int t0 = t_begin; t0 < t_end; t0 += kWgBK) {
    store();
    __syncthreads();
    if (t0 + kWgBK < t_end) load(t0 + kWgBK);
    if (do_bias && tid < BM) {
#pragma unroll 8
      for (int kk = 0; kk < kWgBK; ++kk) bacc += As[kk][tid];
    }
#pragma unroll 8
    for (int kk = 0; kk < kWgBK; ++kk) {
      float a[TM];
      if constexpr (TM >= 4) {
#pragma unroll
        for (int i = 0; i < TM; i += 4) {
          const float4 v = *reinterpret_cast<const float4*>(&As[kk][ty * TM + i]);
          a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = As[kk][ty * TM + i];
      }
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        acc[i][0] = __fmaf_rn(a[i], b.x, acc[i][0]);
        acc[i][1] = __fmaf_rn(a[i], b.y, acc[i][1]);
        acc[i][2] = __fmaf_rn(a[i], b.z, acc[i][2]);
        acc[i][3] = __fmaf_rn(a[i], b.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
  float* o = out + (int64_t)blockIdx.z * E * H;
  const int h = h0 + tx * 4;
  if (h < H) {
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int e = e0 + ty * TM + i;
      if (e < E) *reinterpret_cast<float4*>(o + (int64_t)e * H + h) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
  }
  if (do_bias && tid < BM && e0 + tid < E) bias_out[(int64_t)blockIdx.z * E + e0 + tid] = bacc;
}

// out[i] = sum_{z < S} part[z * n + i], slice order. n4: n / 4 (vectorised) when n % 4 == 0.
__global__ void __launch_bounds__(256) sum_slices_kernel(const float* __restrict__ part, int S, int64_t n,
                                                         float* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if ((n & 3) == 0) {
    const int64_t n4 = n / 4;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
      float4 a = __ldg(reinterpret_cast<const float4*>(part) + i);
      for (int z = 1; z < S; ++z) {
        const float4 b = __ldg(reinterpret_cast<const float4*>(part + (int64_t)z * n) + i);
        a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
      }
      reinterpret_cast<float4*>(out)[i] = a;
    }
  } else {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      float a = part[i];
      for (int z = 1; z < S; ++z) a += part[(int64_t)z * n + i];
      out[i] = a;
    }
  }
}

// ---------------------------------------------------------------------------------------
// 3. dx[t, h] = sum_e dl[t, e] Wr[e, h] (+ the dispatch backward's rows), bf16 layers.
// Block tile 64 tokens x 128 columns; thread (ty, tx) holds 8 tokens x 4 columns; 16
// experts per shared-memory stage.
// ---------------------------------------------------------------------------------------
constexpr int kIgBM = 64, kIgBN = 128, kIgBK = 16, kIgThreads = 256;

__global__ void __launch_bounds__(kIgThreads)
    input_grad_kernel(const float* __restrict__ dl, const uint16_t* __restrict__ wr, const uint16_t* __restrict__ dxd,
                      const int32_t* __restrict__ tok_row, int T, int E, int H, int k, int shared, int64_t R,
                      __nv_bfloat16* __restrict__ dx) {
  __shared__ __align__(16) float As[kIgBK][kIgBM + 4];
  __shared__ __align__(16) float Bs[kIgBK][kIgBN];
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int t0 = blockIdx.y * kIgBM, h0 = blockIdx.x * kIgBN;
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  float ra[4];
  uint4 rb;
  auto load = [&](int e0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * kIgThreads, m = idx / kIgBK, kk = idx % kIgBK;
      const int t = t0 + m, e = e0 + kk;
      ra[q] = (t < T && e < E) ? dl[(int64_t)t * E + e] : 0.0f;
    }
    const int kk = tid / (kIgBN / 8), n = (tid % (kIgBN / 8)) * 8;
    const int e = e0 + kk, h = h0 + n;
    rb = (e < E && h < H) ? __ldg(reinterpret_cast<const uint4*>(wr + (int64_t)e * H + h)) : make_uint4(0u, 0u, 0u, 0u);
  };
  load(0);
  for (int e0 = 0; e0 < E; e0 += kIgBK) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int idx = tid + q * kIgThreads;
      As[idx % kIgBK][idx / kIgBK] = ra[q];
    }
    {
      const int kk = tid / (kIgBN / 8), n = (tid % (kIgBN / 8)) * 8;
      *reinterpret_cast<float4*>(&Bs[kk][n]) = make_float4(bf16_lo(rb.x), bf16_hi(rb.x), bf16_lo(rb.y), bf16_hi(rb.y));
      *reinterpret_cast<float4*>(&Bs[kk][n + 4]) =
          make_float4(bf16_lo(rb.z), bf16_hi(rb.z), bf16_lo(rb.w), bf16_hi(rb.w));
    }
    __syncthreads();
    if (e0 + kIgBK < E) load(e0 + kIgBK);
#pragma unroll
    for (int kk = 0; kk < kIgBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][ty * 8 + 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[i][0] = __fmaf_rn(a[i], b.x, acc[i][0]);
        acc[i][1] = __fmaf_rn(a[i], b.y, acc[i][1]);
        acc[i][2] = __fmaf_rn(a[i], b.z, acc[i][2]);
        acc[i][3] = __fmaf_rn(a[i], b.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
  const int h = h0 + tx * 4;
  if (h >= H) return;
  if (dxd != nullptr) {
    // the dispatch backward's rows, in the order j = 0..k-1, then the shared expert's
    for (int j = 0; j <= k; ++j) {
      if (j == k && !shared) break;
      uint2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = t0 + ty * 8 + i;
        if (t < T) {
          const int64_t r = j < k ? (int64_t)tok_row[(int64_t)t * k + j] : R + t;
          v[i] = __ldg(reinterpret_cast<const uint2*>(dxd + r * H + h));
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (t0 + ty * 8 + i < T) {
          acc[i][0] += bf16_lo(v[i].x);
          acc[i][1] += bf16_hi(v[i].x);
          acc[i][2] += bf16_lo(v[i].y);
          acc[i][3] += bf16_hi(v[i].y);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + ty * 8 + i;
    if (t >= T) continue;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i][0], acc[i][1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i][2], acc[i][3]);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t*>(&lo);
    o.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dx + (int64_t)t * H + h) = o;
  }
}

// 3'. The same sum for few experts (E <= 16), one 128-thread block per token: each thread
// takes 16-byte vectors of 8 columns, issues the NR dispatch rows' loads first, then adds
// dl[t, e] W_router[e] over e (W_router stays in L1) and the rows, in the order of
// input_grad_kernel (experts ascending, then rows j = 0..NR-1), so the bits are the same.
// NR = 0: the router's share alone.
template <int NR>
__global__ void __launch_bounds__(128)
    input_grad_small_kernel(const float* __restrict__ dl, const uint4* __restrict__ wr, const uint4* __restrict__ dxd,
                            const int32_t* __restrict__ tok_row, int E, int H, int k, int64_t R,
                            uint4* __restrict__ dx) {
  __shared__ float dls[16];
  __shared__ int64_t rows[NR > 0 ? NR : 1];
  const int t = blockIdx.x;
  if (threadIdx.x < E) dls[threadIdx.x] = dl[(int64_t)t * E + threadIdx.x];
  if (NR > 0 && threadIdx.x < NR) {
    const int j = threadIdx.x;
    rows[j] = j < k ? (int64_t)tok_row[(int64_t)t * k + j] : R + t;
  }
  __syncthreads();
  const int n8 = H / 8;
  for (int c = threadIdx.x; c < n8; c += 128) {
    uint4 raw[NR > 0 ? NR : 1];
#pragma unroll
    for (int j = 0; j < NR; ++j) raw[j] = __ldg(dxd + rows[j] * n8 + c);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int e = 0; e < E; ++e) {
      const float a = dls[e];
      const uint4 w = __ldg(wr + (int64_t)e * n8 + c);
      const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fmaf_rn(a, bf16_lo(w4[q]), acc[2 * q]);
        acc[2 * q + 1] = __fmaf_rn(a, bf16_hi(w4[q]), acc[2 * q + 1]);
      }
    }
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const uint32_t v4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] += bf16_lo(v4[q]);
        acc[2 * q + 1] += bf16_hi(v4[q]);
      }
    }
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      op[q] = *reinterpret_cast<const uint32_t*>(&p);
    }
    dx[(int64_t)t * n8 + c] = o;
  }
}

}  // namespace

int router_bias_slices(const moe_config_t& c) { return (int)std::max<int64_t>(1, ceil_div(c.T, kBiasSlice)); }

void router_tc_slices(const moe_config_t& c, int* slice, int* slices) {
  // SMs one token slice occupies (CTA pairs of 256 rows when E allows, else single CTAs of
  // 128), and as many slices as fill the 152 SMs, each a whole number of 64-token K stages
  const int64_t sms = (c.E % 256 == 0 ? 2 * (c.E / 256) : c.E / 128) * (int64_t)std::max(1, c.H / 256);
  int64_t s = std::max<int64_t>(1, 152 / std::max<int64_t>(1, sms));
  s = std::min<int64_t>(s, std::max<int64_t>(1, ceil_div(c.T, 64)));
  s = std::min<int64_t>(s, 255);
  const int64_t len = std::max<int64_t>(64, ceil_div(ceil_div(c.T, s), 64) * 64);
  *slice = (int)len;
  *slices = (int)std::max<int64_t>(1, ceil_div(c.T, len));
}

int router_wgrad_slices(const moe_config_t& c) {
  const int bm = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
  const int64_t tiles = ceil_div(c.H, kWgBN) * ceil_div(c.E, bm);
  // about eight blocks per SM of a 152-SM part (enough loads in flight when the product is
  // HBM-bound, several waves when it is ALU-bound), and no slice shorter than 128 tokens
  int64_t s = ceil_div(8 * 152, tiles);
  s = std::min<int64_t>(s, std::max<int64_t>(1, c.T / 128));
  return (int)std::max<int64_t>(1, std::min<int64_t>(s, 64));
}

bool router_backward_tc(const moe_config_t& c) {
  return tc::router_backward_tc_supported(c) && combine_extra_supported(c);
}

namespace {

// token slices of the split reductions: (slice length, slices used)
void slices_of(const moe_config_t& c, int* slice, int* used) {
  const int S = router_wgrad_slices(c);
  *slice = (int)(ceil_div(ceil_div(c.T, S), kWgBK) * kWgBK);
  *used = (int)ceil_div(c.T, *slice);  // <= S
}

// d_bias = column sums of dl: slices of kBiasSlice tokens, then one block over the slices.
cudaError_t bias_grad(const moe_config_t& c, const float* dl, float* d_bias, float* bias_part, cudaStream_t s) {
  const int used = (int)ceil_div(c.T, kBiasSlice);
  colsum_kernel<<<used, 256, 0, s>>>(dl, c.T, c.E, kBiasSlice, used > 1 ? bias_part : d_bias);
  if (used > 1) colsum_kernel<<<1, 256, 0, s>>>(bias_part, used, c.E, used, d_bias);
  return cudaGetLastError();
}

cudaError_t simt_wgrad(const moe_config_t& c, const float* dl, const void* x, float* dw_router, float* d_bias,
                       float* part, float* bias_part, cudaStream_t s) {
  int slice, used;
  slices_of(c, &slice, &used);
  float* out = used > 1 ? part : dw_router;
  float* bout = d_bias ? (used > 1 ? bias_part : d_bias) : nullptr;
  const bool bf = c.act_dtype == MOE_DTYPE_BF16;
  const int bm = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
  const dim3 grid((unsigned)ceil_div(c.H, kWgBN), (unsigned)ceil_div(c.E, bm), (unsigned)used);
#define MOE_WG(BM)                                                                                     \
  if (bf) wgrad_kernel<BM, true><<<grid, kWgThreads, 0, s>>>(dl, x, c.T, c.E, c.H, slice, out, bout); \
  else wgrad_kernel<BM, false><<<grid, kWgThreads, 0, s>>>(dl, x, c.T, c.E, c.H, slice, out, bout)
  if (bm == 8) { MOE_WG(8); }
  else if (bm == 16) { MOE_WG(16); }
  else if (bm == 32) { MOE_WG(32); }
  else { MOE_WG(64); }
#undef MOE_WG
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || used == 1) return e;
  const int64_t n = (int64_t)c.E * c.H;
  const int blocks = (int)std::min<int64_t>(ceil_div(n / 4, 256), 152 * 8);
  sum_slices_kernel<<<blocks, 256, 0, s>>>(part, used, n, dw_router);
  if (d_bias) colsum_kernel<<<1, 256, 0, s>>>(bias_part, used, c.E, used, d_bias);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_backward(const moe_config_t& c, const float* logits, const int32_t* topk_idx,
                                   const float* dtopk_w, const int32_t* counts, float aux_alpha, const void* x,
                                   float* dl, float* dw_router, float* d_bias, const RouterScratch& sc,
                                   DeviceStatus* st, cudaStream_t s) {
  if (c.T == 0) {  // no tokens: zero gradients
    cudaError_t e = dw_router ? cudaMemsetAsync(dw_router, 0, (size_t)c.E * c.H * 4, s) : cudaSuccess;
    if (e == cudaSuccess && d_bias) e = cudaMemsetAsync(d_bias, 0, (size_t)c.E * 4, s);
    return e;
  }
  const bool tc_path = router_backward_tc(c);
  const float a0 = counts ? (float)((double)aux_alpha * c.E / ((double)c.T * c.T * c.k)) : 0.0f;
  const dim3 grid((unsigned)ceil_div(c.T, kLgWarps));
  const int epl = (int)ceil_div(c.E, 32);
  __nv_bfloat16* dlb = tc_path ? static_cast<__nv_bfloat16*>(sc.dl_bf16) : nullptr;
  int tslice = 0, tslices = 1;
  if (tc_path) router_tc_slices(c, &tslice, &tslices);
  int32_t* soff = (tc_path && dw_router && tslices > 1) ? sc.slice_offsets : nullptr;
#define MOE_LG(N)                                                                                              \
  logit_grad_kernel<N><<<grid, kLgWarps * 32, 0, s>>>(logits, topk_idx, dtopk_w, c.T, c.E, c.k, c.score_fn,     \
                                                       c.renorm, c.routed_scale, counts, a0, dl, dlb, soff, tslice,  \
                                                       tslices, st)
  if (epl <= 1) MOE_LG(1);
  else if (epl <= 2) MOE_LG(2);
  else if (epl <= 4) MOE_LG(4);
  else if (epl <= 8) MOE_LG(8);
  else MOE_LG(16);
#undef MOE_LG
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !dw_router) return e;
  if (!tc_path) return simt_wgrad(c, dl, x, dw_router, d_bias, sc.part, sc.bias_part, s);
  if (tslices > 1) {  // K split over token slices, then their partial sums in slice order
    e = tc::launch_router_products(c, dlb, x, nullptr, sc.part, nullptr, st, s, soff, tslices);
    if (e == cudaSuccess) {
      const int64_t n = (int64_t)c.E * c.H;
      const int blocks = (int)std::min<int64_t>(ceil_div(n / 4, 256), 152 * 8);
      sum_slices_kernel<<<blocks, 256, 0, s>>>(sc.part, tslices, n, dw_router);
      e = cudaGetLastError();
    }
  } else {
    e = tc::launch_router_products(c, dlb, x, nullptr, dw_router, nullptr, st, s);
  }
  if (e == cudaSuccess && d_bias) e = bias_grad(c, dl, d_bias, sc.bias_part, s);
  return e;
}

cudaError_t launch_router_input_grad(const moe_config_t& c, const float* dl, const void* dl_bf16,
                                     const void* w_router, const void* dxd, const int32_t* tok_row, void* dx,
                                     const RouterScratch& sc, DeviceStatus* st, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (router_backward_tc(c)) {
    // dx_r = dl W_router on the tensor cores, then dx = the dispatch rows + dx_r
    cudaError_t e = cudaSuccess;
    if (!dl_bf16) {
      const int64_t n = (int64_t)c.T * c.E;
      to_bf16_kernel<<<(unsigned)std::min<int64_t>(ceil_div(n, 256), 152 * 8), 256, 0, s>>>(
          dl, n, static_cast<__nv_bfloat16*>(sc.dl_bf16));
      e = cudaGetLastError();
      dl_bf16 = sc.dl_bf16;
    }
    void* dx_r = dxd ? sc.dx_r : dx;
    if (e == cudaSuccess) e = tc::launch_router_products(c, dl_bf16, nullptr, w_router, nullptr, dx_r, st, s);
    if (e == cudaSuccess && dxd) e = launch_combine_extra(c, dxd, tok_row, dx_r, dx, s);
    return e;
  }
  const int nr = dxd ? c.k + (c.n_shared ? 1 : 0) : 0;
  if (c.E <= 16 && nr <= 9) {
    const uint4* wr = static_cast<const uint4*>(w_router);
    const uint4* rows = static_cast<const uint4*>(dxd);
    uint4* out = static_cast<uint4*>(dx);
#define MOE_IGS(N)                                                                                         \
  case N:                                                                                                  \
    input_grad_small_kernel<N><<<c.T, 128, 0, s>>>(dl, wr, rows, tok_row, c.E, c.H, c.k, routed_rows(c), out); \
    return cudaGetLastError();
    switch (nr) {
      MOE_IGS(0) MOE_IGS(1) MOE_IGS(2) MOE_IGS(3) MOE_IGS(4) MOE_IGS(5) MOE_IGS(6) MOE_IGS(7) MOE_IGS(8) MOE_IGS(9)
      default: break;
    }
#undef MOE_IGS
  }
  const dim3 grid((unsigned)ceil_div(c.H, kIgBN), (unsigned)ceil_div(c.T, kIgBM));
  input_grad_kernel<<<grid, kIgThreads, 0, s>>>(dl, (const uint16_t*)w_router, (const uint16_t*)dxd, tok_row, c.T,
                                                c.E, c.H, c.k, c.n_shared, routed_rows(c), (__nv_bfloat16*)dx);
  return cudaGetLastError();
}

}  // namespace moe
