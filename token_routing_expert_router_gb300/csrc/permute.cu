// S3 dispatch and S7 combine: the on-device form of the dispatch and combine operators
// (Hybrid-EP article: dispatch sends each token only where the routing map says; combine
// brings the expert outputs back with high-precision accumulation). Both walk tokens, so
// x is read once on the way out and y written once on the way back; rows move as 16-byte
// vectors. Also the block quantisers of the FP8 and MXFP8 dispatch variants.
#include "moe_internal.cuh"
#include "mx_common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxVec = 8;  // 16-byte vectors held per thread per pass

// xd[tok_row[t, j]] = x[t] for j < k. One block per token; nvec = 16-byte vectors per row.
__global__ void __launch_bounds__(kThreads) dispatch_kernel(const uint4* __restrict__ x, int nvec,
                                                            int k, const int32_t* __restrict__ tok_row,
                                                            uint4* __restrict__ xd) {
  __shared__ int32_t rows[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) rows[threadIdx.x] = tok_row[(int64_t)t * k + threadIdx.x];
  __syncthreads();
  const uint4* src = x + (int64_t)t * nvec;
  for (int base = 0; base < nvec; base += kThreads * kMaxVec) {
    uint4 v[kMaxVec];
#pragma unroll
    for (int i = 0; i < kMaxVec; ++i) {
      const int idx = base + i * kThreads + threadIdx.x;
      if (idx < nvec) v[i] = __ldg(src + idx);
    }
    for (int j = 0; j < k; ++j) {
      uint4* dst = xd + (int64_t)rows[j] * nvec;
#pragma unroll
      for (int i = 0; i < kMaxVec; ++i) {
        const int idx = base + i * kThreads + threadIdx.x;
        if (idx < nvec) dst[idx] = v[i];
      }
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// e4m3 (round to nearest even, finite values beyond 448 saturate) of four floats, packed
// little-endian (first value in the lowest byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// FP8 dispatch: each token quantised once in 1x128 blocks (one warp per block, four values
// per lane), written to its k rows and, with a shared expert, to row R + t. A pass covers
// 8 warps x kFp8Blocks blocks: each warp issues the loads of its kFp8Blocks blocks before
// quantising any, so several 256-byte loads per warp are in flight; the pass's scales go
// through shared memory and leave with all threads storing, one row's scales per group of
// lanes, instead of one lane per warp issuing a store per block and row.
constexpr int kFp8Blocks = 8;
constexpr int kFp8Warps = 8;
__global__ void __launch_bounds__(32 * kFp8Warps) dispatch_e4m3_kernel(
    const uint2* __restrict__ x, int H, int k, int64_t R, int64_t rows_total, int shared,
    const int32_t* __restrict__ tok_row, uint8_t* __restrict__ xd, float* __restrict__ xd_scale) {
  constexpr int kPass = kFp8Warps * kFp8Blocks;  // blocks per pass
  __shared__ int32_t rows[33];
  __shared__ float sc_s[kPass];
  const int t = blockIdx.x;
  const int nrows = k + shared;
  if (threadIdx.x < k) rows[threadIdx.x] = tok_row[(int64_t)t * k + threadIdx.x];
  if (threadIdx.x == 0 && shared) rows[k] = (int32_t)(R + t);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = H / 128;
  for (int p0 = 0; p0 < nb; p0 += kPass) {  // block-uniform trip count
    uint2 u[kFp8Blocks];
#pragma unroll
    for (int i = 0; i < kFp8Blocks; ++i) {
      const int b = p0 + i * kFp8Warps + warp;
      if (b < nb) u[i] = __ldg(x + ((int64_t)t * H + b * 128) / 4 + lane);
    }
    uint32_t q[kFp8Blocks];
#pragma unroll
    for (int i = 0; i < kFp8Blocks; ++i) {
      q[i] = 0;
      const int b = p0 + i * kFp8Warps + warp;
      if (b >= nb) continue;  // warp-uniform
      const float v0 = bf16_lo(u[i].x), v1 = bf16_hi(u[i].x), v2 = bf16_lo(u[i].y), v3 = bf16_hi(u[i].y);
      float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
      for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      float scale = 1.0f;
      if (amax > 0.0f) {
        scale = __fdiv_rn(amax, 448.0f);
        const float rs = __fdiv_rn(448.0f, amax);
        q[i] = e4m3x4(__fmul_rn(v0, rs), __fmul_rn(v1, rs), __fmul_rn(v2, rs), __fmul_rn(v3, rs));
      }
      if (lane == 0) sc_s[b - p0] = scale;
    }
    for (int j = 0; j < nrows; ++j) {
      const int64_t r = rows[j];
#pragma unroll
      for (int i = 0; i < kFp8Blocks; ++i) {
        const int b = p0 + i * kFp8Warps + warp;
        if (b < nb) reinterpret_cast<uint32_t*>(xd + r * H + b * 128)[lane] = q[i];
      }
    }
    __syncthreads();
    const int npass = min(kPass, nb - p0);
    for (int i = threadIdx.x; i < nrows * npass; i += blockDim.x) {
      const int j = i / npass, bb = i - j * npass;
      xd_scale[(int64_t)(p0 + bb) * rows_total + rows[j]] = sc_s[bb];
    }
    __syncthreads();  // sc_s is rewritten by the next pass
  }
}

// 32 bf16 values from 64 bytes (four 16-byte vectors).
__device__ __forceinline__ void load_bf16x32(const uint4* __restrict__ p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = __ldg(p + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = bf16_lo(w[j]);
      v[8 * i + 2 * j + 1] = bf16_hi(w[j]);
    }
  }
}

// One 1x32 MX block: returns the UE8M0 code and writes the 32 e4m3 codes to q (two 16-byte
// vectors).
__device__ __forceinline__ uint32_t mx_quant_block(const float (&v)[32], uint4 (&q)[2]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int s = mx_scale_exp(amax);
  const float inv = mx_inv_scale(s);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = e4m3x4(__fmul_rn(v[4 * i], inv), __fmul_rn(v[4 * i + 1], inv), __fmul_rn(v[4 * i + 2], inv),
                  __fmul_rn(v[4 * i + 3], inv));
  q[0] = make_uint4(w[0], w[1], w[2], w[3]);
  q[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return (uint32_t)(s + 127);
}

// MXFP8 dispatch: each token quantised once in 1x32 blocks (one block per thread), the
// codes written to its k rows and, with a shared expert, to row R + t; the UE8M0 codes go
// to each row's place in the scale atoms (one 32-bit word per row and 128-column stage).
// A routed row whose expert id is out of range gets its payload but no scales.
__global__ void __launch_bounds__(256) dispatch_mx_kernel(
    const uint4* __restrict__ x, int H, int k, int E, int64_t R, int shared, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ tok_row, const int32_t* __restrict__ offsets, uint8_t* __restrict__ xd,
    uint8_t* __restrict__ xd_sf) {
  extern __shared__ uint32_t codes[];  // [H / 128] words: the token's H / 32 UE8M0 codes
  __shared__ int64_t rows[33];
  __shared__ int64_t atom_row[33];
  __shared__ int32_t atom_i[33];
  const int t = blockIdx.x;
  const int nrows = k + shared;
  if (threadIdx.x < nrows) {
    const int j = threadIdx.x;
    int64_t r, gofs;
    int g;
    if (j < k) {
      r = tok_row[(int64_t)t * k + j];
      g = topk_idx[(int64_t)t * k + j];
      gofs = (g >= 0 && g < E) ? offsets[g] : -1;
    } else {
      r = R + t;
      g = E;
      gofs = R;
    }
    rows[j] = r;
    atom_row[j] = gofs < 0 ? -1 : mx_group_atom_base(gofs, g) + (r - gofs) / 128;
    atom_i[j] = gofs < 0 ? 0 : (int)((r - gofs) % 128);
  }
  __syncthreads();
  const int nb = H / 32;
  uint8_t* code_bytes = reinterpret_cast<uint8_t*>(codes);
  const int lane = threadIdx.x & 31;
  // Every warp quantises 32 consecutive blocks (H % 128 == 0 keeps a warp's blocks all
  // inside the row or all past it); the two 16-byte halves of the blocks are then traded
  // between lanes so that each store instruction writes 512 contiguous bytes.
  for (int b = threadIdx.x; b - lane < nb; b += blockDim.x) {
    const bool live = b < nb;
    uint4 q[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (live) {
      float v[32];
      load_bf16x32(x + ((int64_t)t * H + b * 32) / 8, v);
      code_bytes[b] = (uint8_t)mx_quant_block(v, q);
    }
    // store s (0, 1) of this warp covers its blocks 16 s .. 16 s + 15: lane l writes half
    // l % 2 of block 16 s + l / 2, which lane 16 s + l / 2 holds
    uint4 o[2];
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const int src = 16 * st + (lane >> 1);
      const uint4 h0 = make_uint4(__shfl_sync(0xffffffffu, q[0].x, src), __shfl_sync(0xffffffffu, q[0].y, src),
                                  __shfl_sync(0xffffffffu, q[0].z, src), __shfl_sync(0xffffffffu, q[0].w, src));
      const uint4 h1 = make_uint4(__shfl_sync(0xffffffffu, q[1].x, src), __shfl_sync(0xffffffffu, q[1].y, src),
                                  __shfl_sync(0xffffffffu, q[1].z, src), __shfl_sync(0xffffffffu, q[1].w, src));
      o[st] = (lane & 1) ? h1 : h0;
    }
    const int wb0 = b - lane;  // the warp's first block
    if (wb0 < nb) {
      for (int j = 0; j < nrows; ++j) {
        uint4* dst = reinterpret_cast<uint4*>(xd + rows[j] * H + wb0 * 32);
#pragma unroll
        for (int st = 0; st < 2; ++st)
          if (wb0 + 16 * st + (lane >> 1) < nb) dst[32 * st + lane] = o[st];
      }
    }
  }
  __syncthreads();
  const int ks_total = H / 128;
  for (int i = threadIdx.x; i < nrows * ks_total; i += blockDim.x) {
    const int j = i / ks_total, ks = i - j * ks_total;
    if (atom_row[j] >= 0)
      *reinterpret_cast<uint32_t*>(xd_sf + mx_atom_byte(atom_row[j], ks, ks_total, atom_i[j])) = codes[ks];
  }
}

// MX quantisation of a bf16 [rows, cols] matrix along its rows (offline weight preparation):
// one 1x32 block per thread; rows and cols are multiples of 128; codes to q, UE8M0 scales
// to atoms of 128 rows (tile a = rows [128a, 128a + 128)).
__global__ void __launch_bounds__(256) quantize_mx_kernel(const uint4* __restrict__ src, int64_t rows,
                                                          int64_t cols, uint8_t* __restrict__ q,
                                                          uint8_t* __restrict__ sf) {
  const int64_t nb = cols / 32;
  const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= rows * nb) return;
  const int64_t r = blk / nb, b = blk - r * nb;
  float v[32];
  load_bf16x32(src + (r * cols + b * 32) / 8, v);
  uint4 qq[2];
  const uint32_t code = mx_quant_block(v, qq);
  uint4* dst = reinterpret_cast<uint4*>(q + r * cols + b * 32);
  dst[0] = qq[0];
  dst[1] = qq[1];
  sf[mx_atom_byte(r / 128, (int)(b / 4), (int)(cols / 128), (int)(r % 128)) + (b & 3)] = (uint8_t)code;
}

// y[t] = sum_j w[t,j] * yd[tok_row[t,j]] (+ yd[R+t]), fp32 in fixed j order, one rounding
// to the output type. One block per token, 8 elements per thread per step.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) combine_kernel(const void* __restrict__ yd_, int H, int k,
                                                           const int32_t* __restrict__ tok_row,
                                                           const float* __restrict__ topk_w,
                                                           int shared, int64_t R, void* __restrict__ y_) {
  __shared__ int32_t rows[32];
  __shared__ float wts[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    rows[threadIdx.x] = tok_row[(int64_t)t * k + threadIdx.x];
    wts[threadIdx.x] = topk_w ? topk_w[(int64_t)t * k + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  const int n8 = H / 8;
  for (int c = threadIdx.x; c < n8; c += kThreads) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k + shared; j0 += 8) {
      float v[8][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        if (j < k + shared) {
          const int64_t r = (j < k) ? rows[j] : R + t;
          if (BF16) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(yd_) + (r * H) / 8 + c);
            v[jj][0] = bf16_lo(u.x); v[jj][1] = bf16_hi(u.x);
            v[jj][2] = bf16_lo(u.y); v[jj][3] = bf16_hi(u.y);
            v[jj][4] = bf16_lo(u.z); v[jj][5] = bf16_hi(u.z);
            v[jj][6] = bf16_lo(u.w); v[jj][7] = bf16_hi(u.w);
          } else {
            const float4* p = reinterpret_cast<const float4*>(yd_) + (r * H) / 4 + 2 * c;
            const float4 a = __ldg(p), b = __ldg(p + 1);
            v[jj][0] = a.x; v[jj][1] = a.y; v[jj][2] = a.z; v[jj][3] = a.w;
            v[jj][4] = b.x; v[jj][5] = b.y; v[jj][6] = b.z; v[jj][7] = b.w;
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int j = j0 + jj;
        if (j < k) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(wts[j], v[jj][i], acc[i]);
        } else if (j < k + shared) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], v[jj][i]);
        }
      }
    }
    if (BF16) {
      uint4 o;
      __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
      __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
      o.x = *reinterpret_cast<uint32_t*>(&p0);
      o.y = *reinterpret_cast<uint32_t*>(&p1);
      o.z = *reinterpret_cast<uint32_t*>(&p2);
      o.w = *reinterpret_cast<uint32_t*>(&p3);
      reinterpret_cast<uint4*>(y_)[((int64_t)t * H) / 8 + c] = o;
    } else {
      float4* p = reinterpret_cast<float4*>(y_) + ((int64_t)t * H) / 4 + 2 * c;
      p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

// Same sum with the row count NR = k (+1 shared) known at compile time: every row's
// 16-byte vector of a chunk is loaded before any of them is summed, so one memory round
// trip covers all NR rows. With few rows, each thread takes U chunks per pass and issues
// all NR * U loads first, so about eight 16-byte loads are in flight per thread whatever k
// is. The shared row enters with weight 1 (fma(1, v, acc) == acc + v). EXTRA (bf16): the
// last of the NR rows is row t of a separate [T, H] buffer, added with weight 1 (the
// router's share of the input gradient, after the dispatch backward's rows).
template <int NR, bool BF16, bool EXTRA = false>
__global__ void __launch_bounds__(kThreads) combine_nr_kernel(const void* __restrict__ yd_, int H, int k,
                                                              const int32_t* __restrict__ tok_row,
                                                              const float* __restrict__ topk_w, int64_t R,
                                                              void* __restrict__ y_,
                                                              const void* __restrict__ extra_ = nullptr) {
  constexpr int U = NR >= 8 ? 1 : 8 / NR;
  __shared__ int64_t rows[NR];
  __shared__ float wts[NR];
  const int t = blockIdx.x;
  if (threadIdx.x < NR) {
    const int j = threadIdx.x;
    rows[j] = j < k ? (int64_t)tok_row[(int64_t)t * k + j] : R + t;
    wts[j] = (j < k && topk_w) ? topk_w[(int64_t)t * k + j] : 1.0f;
  }
  __syncthreads();
  const int n8 = H / 8;
  for (int base = threadIdx.x; base < n8; base += kThreads * U) {
    if (BF16) {
      uint4 raw[U][NR];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * kThreads;
        if (c < n8) {
#pragma unroll
          for (int j = 0; j < NR; ++j)
            raw[u][j] = (EXTRA && j == NR - 1) ? __ldg(reinterpret_cast<const uint4*>(extra_) + (int64_t)t * n8 + c)
                                               : __ldg(reinterpret_cast<const uint4*>(yd_) + rows[j] * n8 + c);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * kThreads;
        if (c >= n8) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const float wj = wts[j];
          const uint32_t w4[4] = {raw[u][j].x, raw[u][j].y, raw[u][j].z, raw[u][j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[2 * q] = __fmaf_rn(wj, bf16_lo(w4[q]), acc[2 * q]);
            acc[2 * q + 1] = __fmaf_rn(wj, bf16_hi(w4[q]), acc[2 * q + 1]);
          }
        }
        uint4 o;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        o.z = *reinterpret_cast<uint32_t*>(&p2);
        o.w = *reinterpret_cast<uint32_t*>(&p3);
        reinterpret_cast<uint4*>(y_)[(int64_t)t * n8 + c] = o;
      }
    } else {
      float4 raw[U][NR][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * kThreads;
        if (c < n8) {
#pragma unroll
          for (int j = 0; j < NR; ++j) {
            const float4* p = reinterpret_cast<const float4*>(yd_) + rows[j] * (H / 4) + 2 * c;
            raw[u][j][0] = __ldg(p);
            raw[u][j][1] = __ldg(p + 1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = base + u * kThreads;
        if (c >= n8) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          const float wj = wts[j];
          acc[0] = __fmaf_rn(wj, raw[u][j][0].x, acc[0]); acc[1] = __fmaf_rn(wj, raw[u][j][0].y, acc[1]);
          acc[2] = __fmaf_rn(wj, raw[u][j][0].z, acc[2]); acc[3] = __fmaf_rn(wj, raw[u][j][0].w, acc[3]);
          acc[4] = __fmaf_rn(wj, raw[u][j][1].x, acc[4]); acc[5] = __fmaf_rn(wj, raw[u][j][1].y, acc[5]);
          acc[6] = __fmaf_rn(wj, raw[u][j][1].z, acc[6]); acc[7] = __fmaf_rn(wj, raw[u][j][1].w, acc[7]);
        }
        float4* p = reinterpret_cast<float4*>(y_) + ((int64_t)t * H) / 4 + 2 * c;
        p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
    }
  }
}

// Combine backward, one block per token: dy[t] is read once per row it feeds;
// dyd[tok_row[t,j]] = bf16(w[t,j] * dy[t]), dyd[R+t] = dy[t] (shared expert), and
// dtopk_w[t,j] = sum_o dy[t,o] * yd[tok_row[t,j], o] in fp32 (block reduction).
__global__ void __launch_bounds__(kThreads) combine_backward_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ yd, int H, int k, const int32_t* __restrict__ tok_row,
    const float* __restrict__ topk_w, int shared, int64_t R, uint4* __restrict__ dyd, float* __restrict__ dtopk_w) {
  __shared__ int64_t rows[32];
  __shared__ float wts[32];
  __shared__ float red[32][kThreads / 32];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < k) {
    rows[threadIdx.x] = tok_row[(int64_t)t * k + threadIdx.x];
    wts[threadIdx.x] = topk_w[(int64_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int n8 = H / 8;
  const uint4* g = dy + (int64_t)t * n8;
  for (int j = 0; j < k; ++j) {
    const float wj = wts[j];
    const uint4* src = yd + rows[j] * n8;
    uint4* dst = dyd + rows[j] * n8;
    float dot = 0.0f;
    for (int c = threadIdx.x; c < n8; c += kThreads) {
      const uint4 a = __ldg(g + c), b = __ldg(src + c);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a0 = bf16_lo(av[q]), a1 = bf16_hi(av[q]);
        dot = __fmaf_rn(a0, bf16_lo(bv[q]), dot);
        dot = __fmaf_rn(a1, bf16_hi(bv[q]), dot);
        const __nv_bfloat162 p = __floats2bfloat162_rn(wj * a0, wj * a1);
        o[q] = *reinterpret_cast<const uint32_t*>(&p);
      }
      dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) red[j][warp] = dot;
  }
  if (shared) {
    uint4* dst = dyd + (R + t) * n8;
    for (int c = threadIdx.x; c < n8; c += kThreads) dst[c] = __ldg(g + c);
  }
  __syncthreads();
  if (threadIdx.x < k) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += red[threadIdx.x][w];
    dtopk_w[(int64_t)t * k + threadIdx.x] = s;
  }
}

template <int NR>
cudaError_t launch_combine_nr(const moe_config_t& c, const void* yd, const int32_t* tok_row,
                              const float* topk_w, void* y, cudaStream_t s) {
  if (c.act_dtype == MOE_DTYPE_BF16)
    combine_nr_kernel<NR, true><<<c.T, kThreads, 0, s>>>(yd, c.H, c.k, tok_row, topk_w, routed_rows(c), y);
  else
    combine_nr_kernel<NR, false><<<c.T, kThreads, 0, s>>>(yd, c.H, c.k, tok_row, topk_w, routed_rows(c), y);
  return cudaGetLastError();
}

// Block quantisation of a bf16 matrix (br x bc blocks) with the dispatch rule.
__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t* __restrict__ src, int64_t rows,
                                                       int64_t cols, int br, int bc, uint8_t* __restrict__ q,
                                                       float* __restrict__ scale) {
  __shared__ float red[8];
  const int64_t nbc = ceil_div(cols, bc);
  const int64_t r0 = (blockIdx.x / nbc) * br, c0 = (blockIdx.x % nbc) * bc;
  const int64_t r1 = min(r0 + br, rows), c1 = min(c0 + bc, cols);
  const int64_t w = c1 - c0, n = (r1 - r0) * w;
  float amax = 0.0f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t r = r0 + i / w, c = c0 + i % w;
    amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)src[r * cols + c] << 16)));
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.0f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
  const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const float rs = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 0.0f;
  if (threadIdx.x == 0) scale[blockIdx.x] = sc;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t r = r0 + i / w, c = c0 + i % w;
    const float v = __uint_as_float((uint32_t)src[r * cols + c] << 16);
    const __nv_fp8_storage_t code = __nv_cvt_float_to_fp8(__fmul_rn(v, rs), __NV_SATFINITE, __NV_E4M3);
    q[r * cols + c] = amax > 0.0f ? (uint8_t)code : (uint8_t)0;
  }
}

}  // namespace

cudaError_t launch_dispatch(const moe_config_t& c, const void* x, const int32_t* tok_row,
                            void* xd, float* xd_scale, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (c.xfer_dtype == MOE_DTYPE_E4M3) {
    dispatch_e4m3_kernel<<<c.T, 32 * kFp8Warps, 0, s>>>(reinterpret_cast<const uint2*>(x), c.H, c.k,
                                             routed_rows(c), total_rows(c), c.n_shared ? 1 : 0,
                                             tok_row, reinterpret_cast<uint8_t*>(xd), xd_scale);
  } else {
    const int esize = c.act_dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const int nvec = c.H * esize / 16;
    dispatch_kernel<<<c.T, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(x), nvec, c.k, tok_row,
                                              reinterpret_cast<uint4*>(xd));
  }
  return cudaGetLastError();
}

template <int NR>
cudaError_t launch_combine_extra_nr(const moe_config_t& c, const void* yd, const int32_t* tok_row, const void* extra,
                                    void* y, cudaStream_t s) {
  combine_nr_kernel<NR, true, true><<<c.T, kThreads, 0, s>>>(yd, c.H, c.k, tok_row, nullptr, routed_rows(c), y, extra);
  return cudaGetLastError();
}

bool combine_extra_supported(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.k + (c.n_shared ? 1 : 0) + 1 <= 10;
}

cudaError_t launch_combine_extra(const moe_config_t& c, const void* yd, const int32_t* tok_row, const void* extra,
                                 void* y, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  switch (c.k + (c.n_shared ? 1 : 0) + 1) {
    case 2: return launch_combine_extra_nr<2>(c, yd, tok_row, extra, y, s);
    case 3: return launch_combine_extra_nr<3>(c, yd, tok_row, extra, y, s);
    case 4: return launch_combine_extra_nr<4>(c, yd, tok_row, extra, y, s);
    case 5: return launch_combine_extra_nr<5>(c, yd, tok_row, extra, y, s);
    case 6: return launch_combine_extra_nr<6>(c, yd, tok_row, extra, y, s);
    case 7: return launch_combine_extra_nr<7>(c, yd, tok_row, extra, y, s);
    case 8: return launch_combine_extra_nr<8>(c, yd, tok_row, extra, y, s);
    case 9: return launch_combine_extra_nr<9>(c, yd, tok_row, extra, y, s);
    case 10: return launch_combine_extra_nr<10>(c, yd, tok_row, extra, y, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine(const moe_config_t& c, const void* yd, const int32_t* tok_row,
                           const float* topk_w, void* y, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int shared = c.n_shared ? 1 : 0;
  switch (c.k + shared) {
    case 1: return launch_combine_nr<1>(c, yd, tok_row, topk_w, y, s);
    case 2: return launch_combine_nr<2>(c, yd, tok_row, topk_w, y, s);
    case 3: return launch_combine_nr<3>(c, yd, tok_row, topk_w, y, s);
    case 4: return launch_combine_nr<4>(c, yd, tok_row, topk_w, y, s);
    case 5: return launch_combine_nr<5>(c, yd, tok_row, topk_w, y, s);
    case 6: return launch_combine_nr<6>(c, yd, tok_row, topk_w, y, s);
    case 7: return launch_combine_nr<7>(c, yd, tok_row, topk_w, y, s);
    case 8: return launch_combine_nr<8>(c, yd, tok_row, topk_w, y, s);
    case 9: return launch_combine_nr<9>(c, yd, tok_row, topk_w, y, s);
    default: break;  // larger k: the generic loop below
  }
  if (c.act_dtype == MOE_DTYPE_BF16)
    combine_kernel<true><<<c.T, kThreads, 0, s>>>(yd, c.H, c.k, tok_row, topk_w, shared, routed_rows(c), y);
  else
    combine_kernel<false><<<c.T, kThreads, 0, s>>>(yd, c.H, c.k, tok_row, topk_w, shared, routed_rows(c), y);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_mx(const moe_config_t& c, const void* x, const int32_t* topk_idx,
                               const int32_t* tok_row, const int32_t* offsets, void* xd, void* xd_sf,
                               cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const size_t smem = align_up((size_t)c.H / 32, 16);
  dispatch_mx_kernel<<<c.T, 256, smem, s>>>(reinterpret_cast<const uint4*>(x), c.H, c.k, c.E, routed_rows(c),
                                            c.n_shared ? 1 : 0, topk_idx, tok_row, offsets,
                                            reinterpret_cast<uint8_t*>(xd), reinterpret_cast<uint8_t*>(xd_sf));
  return cudaGetLastError();
}

cudaError_t launch_quantize_mx(const void* src, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                               cudaStream_t s) {
  const int64_t nblk = rows * (cols / 32);
  if (nblk == 0) return cudaSuccess;
  quantize_mx_kernel<<<(unsigned)ceil_div(nblk, 256), 256, 0, s>>>(reinterpret_cast<const uint4*>(src), rows, cols,
                                                                    q, sf);
  return cudaGetLastError();
}

cudaError_t launch_combine_backward(const moe_config_t& c, const void* dy, const void* yd, const int32_t* tok_row,
                                    const float* topk_w, void* dyd, float* dtopk_w, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  combine_backward_kernel<<<c.T, kThreads, 0, s>>>(reinterpret_cast<const uint4*>(dy), reinterpret_cast<const uint4*>(yd),
                                                   c.H, c.k, tok_row, topk_w, c.n_shared ? 1 : 0, routed_rows(c),
                                                   reinterpret_cast<uint4*>(dyd), dtopk_w);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* src, int64_t rows, int64_t cols, int br, int bc,
                                 uint8_t* q, float* scale, cudaStream_t s) {
  const int64_t nblk = ceil_div(rows, br) * ceil_div(cols, bc);
  if (nblk == 0) return cudaSuccess;
  quantize_kernel<<<(unsigned)nblk, 256, 0, s>>>(reinterpret_cast<const uint16_t*>(src), rows, cols,
                                                 br, bc, q, scale);
  return cudaGetLastError();
}

}  // namespace moe
