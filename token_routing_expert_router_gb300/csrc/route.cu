// S1 (score + top-k, group-limited selection, weights) and S2 (per-expert counts, offsets
// and the stable permutation) of the MoE layer forward.
//
// The router activates k experts per token ("Scalable Training of Mixture-of-Experts Models
// with Megatron Core" summary, "O essencial"); the dispatch follows the routing map
// (Hybrid-EP article); the per-expert shapes stay in device memory so no host sync is
// needed (Megatron-Core summary, section 2.4, device-initiated kernels).
#include <float.h>
#include <limits.h>

#include <algorithm>

#include "moe_internal.cuh"
#include "tc_common.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Deterministic fp32 exp: Cody-Waite reduction by ln 2 split into a 16-bit head and a
// tail, a degree-7 Taylor polynomial of e^r (|r| <= ln2/2) by Horner with fused
// multiply-adds, and a two-step power-of-two scaling. Written with explicit round-to-
// nearest intrinsics so that no contraction or fast path changes a bit: any IEEE machine
// running the same operations gets the same result, which is what lets group-limited
// routing decide the same groups everywhere. Constants are the fp32 bit patterns of
// 1/ln2, ln2 (head, tail) and 1/i!.
__device__ __forceinline__ float det_exp(float a) {
  if (a != a) return a;
  if (a > __int_as_float(0x42b17218)) return __int_as_float(0x7f800000);  // > 88.7228...
  if (a < __int_as_float(0xc2cff1b5)) return 0.0f;                        // < -103.972...
  const float n = rintf(__fmul_rn(a, __int_as_float(0x3fb8aa3b)));
  float r = __fmaf_rn(-n, __int_as_float(0x3f317200), a);
  r = __fmaf_rn(-n, __int_as_float(0x35bfbe8e), r);
  float p = __int_as_float(0x39500d01);             // 1/7!
  p = __fmaf_rn(p, r, __int_as_float(0x3ab60b61));  // 1/6!
  p = __fmaf_rn(p, r, __int_as_float(0x3c088889));  // 1/5!
  p = __fmaf_rn(p, r, __int_as_float(0x3d2aaaab));  // 1/4!
  p = __fmaf_rn(p, r, __int_as_float(0x3e2aaaab));  // 1/3!
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int ni = (int)n;
  const int n1 = ni >> 1, n2 = ni - n1;
  return __fmul_rn(__fmul_rn(p, __int_as_float((n1 + 127) << 23)), __int_as_float((n2 + 127) << 23));
}

__device__ __forceinline__ float det_sigmoid(float l) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, det_exp(-l)));
}

// (key, idx) order: larger key first, equal keys to the lower index.
__device__ __forceinline__ bool better(float k1, int i1, float k2, int i2) {
  return k1 > k2 || (k1 == k2 && i1 < i2);
}

// Order-preserving integer image of a finite float (larger float, larger key; -0 and +0
// both map to +0's key). Every image is nonzero, so 0 can mark an empty slot.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x == 0.0f ? 0.0f : x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

__device__ __forceinline__ void warp_argmax(float& key, int& idx) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float ok = __shfl_xor_sync(kFull, key, off);
    const int oi = __shfl_xor_sync(kFull, idx, off);
    if (better(ok, oi, key, idx)) { key = ok; idx = oi; }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

// Token t's logits into the warp's registers: lane l gets experts l, l+32, ... (NSLOT slots;
// slots past E hold -FLT_MAX). Issued apart from route_token so that a warp can load its
// next token while it routes this one.
template <int NSLOT>
__device__ __forceinline__ void load_logits(const float* __restrict__ logits, int t, int E, float (&x)[NSLOT]) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + (int64_t)t * E;
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) {
    const int e = s * 32 + lane;
    x[s] = e < E ? row[e] : -FLT_MAX;
  }
}

// S1 for one token t, by one warp, from its logits x (load_logits): lane l holds experts l,
// l+32, l+64, ... (NSLOT slots). Writes the token's k expert ids and weights and returns, in
// lane j < k, the token's j-th expert. sc: this warp's E floats of shared memory (group-limited
// routing whose groups are not single slots).
template <int NSLOT>
__device__ __forceinline__ int route_token(const float (&x)[NSLOT], int t, int E, int k, int score_fn,
                                           int renorm, int G, int g_keep, int group_score, float rho,
                                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* sc,
                                           DeviceStatus* st) {
  const int lane = threadIdx.x & 31;

  float v[NSLOT];
  uint32_t ok = 0;
  bool bad = false;
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) {
    v[s] = -FLT_MAX;
    if (s * 32 + lane < E) {
      float xv = x[s];
      if (!isfinite(xv)) { bad = true; xv = -FLT_MAX; }
      v[s] = xv;
      ok |= 1u << s;
    }
  }
  if (__any_sync(kFull, bad) && lane == 0) set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);

  uint32_t allowed = ok;
  if (G > 1 && g_keep < G) {
    uint32_t keep = 0;
    if (E == 32 * G) {
      // One group per slot (group g = experts 32g .. 32g + 31 = slot g): each group's key
      // comes from warp reductions of its 32 scores. Scores are >= +0 (a sigmoid), so their
      // bit patterns order as unsigned integers; the second largest equals the largest when
      // two lanes hold it.
      float gk[NSLOT];
#pragma unroll
      for (int s = 0; s < NSLOT; ++s) {
        gk[s] = -INFINITY;
        if (s < G) {
          const uint32_t b = __float_as_uint(det_sigmoid(v[s]));
          const uint32_t m1 = __reduce_max_sync(kFull, b);
          float g = __uint_as_float(m1);
          if (group_score == MOE_GROUP_SCORE_TOP2_SUM) {
            uint32_t m2 = m1;
            if (__popc(__ballot_sync(kFull, b == m1)) < 2) m2 = __reduce_max_sync(kFull, b == m1 ? 0u : b);
            g = __fadd_rn(g, __uint_as_float(m2));
          }
          gk[s] = g;
        }
      }
      // the g_keep best groups in (key, index) order: those with fewer than g_keep better ones
#pragma unroll
      for (int g = 0; g < NSLOT; ++g) {
        int rank = 0;
#pragma unroll
        for (int h = 0; h < NSLOT; ++h)
          rank += (h < G && better(gk[h], h, gk[g], g)) ? 1 : 0;
        if (g < G && rank < g_keep) keep |= 1u << g;
      }
      allowed = ok & keep;
    } else {
#pragma unroll
      for (int s = 0; s < NSLOT; ++s)
        if (ok >> s & 1) sc[s * 32 + lane] = det_sigmoid(v[s]);
      __syncwarp();
      const int gs = E / G;
      float gkey = -INFINITY;
      int gidx = INT_MAX;
      if (lane < G) {
        float m1 = -INFINITY, m2 = -INFINITY;  // the two largest scores of the group
        // lanes start at different offsets of their groups (no bank conflicts); the two
        // largest do not depend on the order the scores are visited in
        for (int i = 0; i < gs; ++i) {
          const float x = sc[lane * gs + (i + lane) % gs];
          if (x > m1) { m2 = m1; m1 = x; }
          else if (x > m2) m2 = x;
        }
        gkey = (group_score == MOE_GROUP_SCORE_TOP2_SUM && gs >= 2) ? __fadd_rn(m1, m2) : m1;
        gidx = lane;
      }
      __syncwarp();  // the scores are read before the warp's next token overwrites them
      for (int r = 0; r < g_keep; ++r) {
        float bk = gkey;
        int bi = gidx;
        warp_argmax(bk, bi);
        keep |= 1u << bi;
        if (lane == bi) { gkey = -INFINITY; gidx = INT_MAX; }
      }
      allowed = 0;
#pragma unroll
      for (int s = 0; s < NSLOT; ++s) {
        const int e = s * 32 + lane;
        if ((ok >> s & 1) && (keep >> (e / gs) & 1)) allowed |= 1u << s;
      }
    }
  }

  // Top-k by (logit, index): each round takes the warp's largest key (one reduction), then
  // the lowest expert index holding it (a second one); only the lane that held the winner
  // moves on to its next best slot. Keys are the logits' order-preserving integer images,
  // with -0 taken as +0 so that equal logits tie; 0 marks a slot that is out of the race.
  uint32_t key[NSLOT];
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) key[s] = order_key(v[s]);
  uint32_t live = allowed;  // the lane's slots still in the race
  uint32_t bk = 0u;
  int bs = 0;
#pragma unroll
  for (int s = 0; s < NSLOT; ++s)
    if ((live >> s & 1) && key[s] > bk) { bk = key[s]; bs = s; }
  int my_idx = 0;
  uint32_t my_k = 0u;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(kFull, bk);
    const uint32_t cand = (bk == m && bk != 0u) ? (uint32_t)(bs * 32 + lane) : 0xffffffffu;
    const uint32_t bi = __reduce_min_sync(kFull, cand);
    if (lane == j) { my_idx = (int)bi; my_k = m; }
    if (cand == bi) {  // this lane's best was taken
      live &= ~(1u << bs);
      bk = 0u;
      bs = 0;
#pragma unroll
      for (int s = 0; s < NSLOT; ++s)
        if ((live >> s & 1) && key[s] > bk) { bk = key[s]; bs = s; }
    }
  }
  const float my_key = key_value(my_k);

  float w;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    uint32_t mk = 0u;
#pragma unroll
    for (int s = 0; s < NSLOT; ++s)
      if (ok >> s & 1) mk = max(mk, order_key(v[s]));
    const float m = key_value(__reduce_max_sync(kFull, mk));
    const float ej = (lane < k) ? expf(my_key - m) : 0.0f;
    float part = 0.0f;
    if (renorm) {
      part = ej;
    } else {
#pragma unroll
      for (int s = 0; s < NSLOT; ++s)
        if (ok >> s & 1) part += expf(v[s] - m);
    }
    w = ej / warp_sum(part);
  } else {
    const float sj = (lane < k) ? det_sigmoid(my_key) : 0.0f;
    const float denom = renorm ? warp_sum(sj) : 1.0f;
    w = sj / denom;
  }
  if (lane < k) {
    topk_idx[(int64_t)t * k + lane] = my_idx;
    topk_w[(int64_t)t * k + lane] = w * rho;
  }
  return my_idx;
}

// ---- S1 for four tokens a warp (E of 64, 128 or 256, k <= 8, no group limit or 8 groups)
// Lane j of 8-lane segment g holds experts [j M, (j + 1) M) of token t + g (M = E / 8; with 8
// groups, group j). One pass over its experts keeps the lane's best 8 in (logit, index)
// order, packed as (order_key << 32 | ~index) so that a larger value is a better expert,
// and with group-limited routing the two largest sigmoid scores of its group. Three
// butterfly steps over the segment then merge the lanes' lists (a bitonic merge of two
// descending lists of 8 keeps their best 8), after which every lane of the segment holds
// the token's best 8 and lane j takes the j-th. No reduction across the 32 lanes per
// selected expert, and four tokens share each instruction: the warp-per-token form spends
// most of its instruction slots on those reductions.
__host__ __device__ inline bool route_sub8(int E, int k, int G, int g_keep) {
  return (E == 64 || E == 128 || E == 256) && k <= 8 && (!(G > 1 && g_keep < G) || G == 8);
}

// A bitonic sequence of 8 sorted descending (half-cleaners of width 4, 2, 1).
__device__ __forceinline__ void bitonic8_desc(uint64_t (&c)[8]) {
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & d) == 0 && c[i + d] > c[i]) {
        const uint64_t tmp = c[i];
        c[i] = c[i + d];
        c[i + d] = tmp;
      }
}

// Sum over the lane's 8-lane segment (a butterfly: every lane gets the same bits).
__device__ __forceinline__ float seg8_sum(float v) {
  v += __shfl_xor_sync(kFull, v, 1);
  v += __shfl_xor_sync(kFull, v, 2);
  v += __shfl_xor_sync(kFull, v, 4);
  return v;
}

// Routes token t (its segment's; `active` false past the warp's tokens) and returns, in
// lane j < k of the segment, the token's j-th expert. logits 16-byte aligned.
template <int M>
__device__ __forceinline__ int route_tokens8(const float* __restrict__ logits, int t, bool active, int E, int k,
                                             int score_fn, int renorm, int G, int g_keep, int group_score, float rho,
                                             int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                             DeviceStatus* st) {
  const int lane = threadIdx.x & 31, j = lane & 7;
  const bool grouped = G > 1 && g_keep < G;
  const float4* row = reinterpret_cast<const float4*>(logits + (int64_t)t * E + j * M);
  uint64_t top[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) top[i] = 0ull;
  uint32_t all_max = 0u;      // the largest key of the lane's experts (the softmax's max)
  uint32_t s1 = 0u, s2 = 0u;  // the two largest sigmoid scores of the lane's group, as bits
  bool bad = false;
  if (active) {
#pragma unroll
    for (int c = 0; c < M / 4; ++c) {
      const float4 q = row[c];
      const float xs[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float x = xs[u];
        if (!isfinite(x)) { bad = true; x = -FLT_MAX; }
        const uint32_t key = order_key(x);
        all_max = max(all_max, key);
        if (grouped) {  // the multiset's two largest: a tie with the largest is the second
          const uint32_t b = __float_as_uint(det_sigmoid(x));
          s2 = max(s2, min(s1, b));
          s1 = max(s1, b);
        }
        const uint64_t pk = (uint64_t)key << 32 | (0xffffffffu - (uint32_t)(j * M + 4 * c + u));
        if (pk > top[7]) {  // insert, keeping the list descending
          top[7] = pk;
#pragma unroll
          for (int i = 7; i > 0; --i)
            if (top[i] > top[i - 1]) {
              const uint64_t tmp = top[i];
              top[i] = top[i - 1];
              top[i - 1] = tmp;
            }
        }
      }
    }
  }
  if (bad) set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);
  if (grouped) {  // 8 groups: the g_keep best in (key, index) order keep their candidates
    const float gk = group_score == MOE_GROUP_SCORE_TOP2_SUM ? __fadd_rn(__uint_as_float(s1), __uint_as_float(s2))
                                                             : __uint_as_float(s1);
    int rank = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) rank += better(__shfl_sync(kFull, gk, (lane & ~7) | i), i, gk, j) ? 1 : 0;
    if (rank >= g_keep)
#pragma unroll
      for (int i = 0; i < 8; ++i) top[i] = 0ull;
  }
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    uint64_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(kFull, (unsigned long long)top[i], off);
#pragma unroll
    for (int i = 0; i < 8; ++i) top[i] = max(top[i], o[7 - i]);
    bitonic8_desc(top);
  }
  uint64_t pj = 0ull;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i == j) pj = top[i];
  const int my_idx = (int)(0xffffffffu - (uint32_t)pj);  // -1 where no candidate is left
  const float my_key = key_value((uint32_t)(pj >> 32));
  float w;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    uint32_t mk = all_max;
    mk = max(mk, __shfl_xor_sync(kFull, mk, 1));
    mk = max(mk, __shfl_xor_sync(kFull, mk, 2));
    mk = max(mk, __shfl_xor_sync(kFull, mk, 4));
    const float m = key_value(mk);
    const float ej = (j < k) ? expf(my_key - m) : 0.0f;
    float part = 0.0f;
    if (renorm) {
      part = ej;
    } else if (active) {
#pragma unroll
      for (int c = 0; c < M / 4; ++c) {
        const float4 q = row[c];
        const float xs[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) part += expf((isfinite(xs[u]) ? xs[u] : -FLT_MAX) - m);
      }
    }
    w = ej / seg8_sum(part);
  } else {
    const float sj = (j < k) ? det_sigmoid(my_key) : 0.0f;
    w = sj / (renorm ? seg8_sum(sj) : 1.0f);
  }
  if (active && j < k) {
    topk_idx[(int64_t)t * k + j] = my_idx;
    topk_w[(int64_t)t * k + j] = w * rho;
  }
  return my_idx;
}

// ---- auxiliary load-balancing loss, summed exactly
// Each token's probabilities (the softmax of its logits over all experts, or its sigmoid
// scores divided by their sum; a non-finite logit counts as -FLT_MAX, as in routing) are
// rounded to multiples of 2^-32 and added as 64-bit integers, so a sum does not depend on
// how the tokens are split between warps, blocks or launches: the single-launch routing and
// moe_aux_loss's own pass give the same bits. kAuxOne = 2^32 stands for probability 1.
constexpr float kAuxOne = 4294967296.0f;

// One token by one warp, from its logits x (load_logits): lane l adds the fixed-point
// probability of experts l, l + 32, ...
template <int NSLOT>
__device__ __forceinline__ void aux_token_fixed(const float (&x)[NSLOT], int E, int score_fn,
                                                uint64_t (&acc)[NSLOT]) {
  const int lane = threadIdx.x & 31;
  float v[NSLOT];
  float m = -FLT_MAX;
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) {
    const int e = s * 32 + lane;
    float xv = -FLT_MAX;
    if (e < E) {
      xv = x[s];
      if (!isfinite(xv)) xv = -FLT_MAX;
    }
    v[s] = xv;
    m = fmaxf(m, xv);
  }
  float sum = 0.0f;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    m = warp_max(m);
#pragma unroll
    for (int s = 0; s < NSLOT; ++s) {
      v[s] = s * 32 + lane < E ? expf(v[s] - m) : 0.0f;
      sum += v[s];
    }
  } else {
#pragma unroll
    for (int s = 0; s < NSLOT; ++s) {
      v[s] = s * 32 + lane < E ? det_sigmoid(v[s]) : 0.0f;
      sum += v[s];
    }
  }
  sum = warp_sum(sum);
  if (!(sum > 0.0f)) return;  // every score zero: the token adds nothing
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) acc[s] += __float2ull_rn(v[s] / sum * kAuxOne);
}

// loss = alpha * E / (T k) * sum_e counts[e] * Pbar_e, Pbar_e = S_e / (2^32 T), from the exact
// V = sum_e counts[e] * S_e (at most 2^31 * 2^63 * 512 < 2^103), in fp32: V over
// T^2 k 2^32 / E, then times alpha (a few roundings, each 2^-24 relative; fp64 arithmetic is
// slow on this part, and the loss is a float). Every path that forms the loss calls this.
__device__ __forceinline__ float aux_loss_from(unsigned __int128 V, float alpha, int E, int T, int k) {
  const float v = __fadd_rn(__fmul_rn((float)(uint64_t)(V >> 64), 18446744073709551616.0f), (float)(uint64_t)V);
  const float d = __fmul_rn(__fmul_rn((float)T, (float)T), __fdiv_rn(__fmul_rn((float)k, 4294967296.0f), (float)E));
  return __fmul_rn(__fdiv_rn(v, d), alpha);
}

// Sum of a 128-bit value over the warp.
__device__ __forceinline__ unsigned __int128 warp_sum_u128(unsigned __int128 v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const uint64_t lo = __shfl_xor_sync(kFull, (unsigned long long)(uint64_t)v, off);
    const uint64_t hi = __shfl_xor_sync(kFull, (unsigned long long)(uint64_t)(v >> 64), off);
    v += ((unsigned __int128)hi << 64) | lo;
  }
  return v;
}

// The block's V (every thread passes its share; blockDim a multiple of 32, at most 1024),
// returned to thread 0. red: 32 shared 128-bit slots.
__device__ __forceinline__ unsigned __int128 block_sum_u128(unsigned __int128 v, unsigned __int128* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u128(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned __int128 t = 0;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
  return t;
}

// One warp per token.
template <int NSLOT>
__global__ void __launch_bounds__(256) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int score_fn, int renorm, int G,
    int g_keep, int group_score, float rho, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, DeviceStatus* st, int sub8) {
  extern __shared__ float s_score[];  // [warps][E] sigmoid scores (group-limited only)
  const int warp = threadIdx.x >> 5;
  if constexpr (NSLOT == 2 || NSLOT == 4 || NSLOT == 8) {
    if (sub8) {  // four tokens a warp, E = 32 NSLOT
      const int tb = (blockIdx.x * (blockDim.x >> 5) + warp) * 4;
      if (tb >= T) return;
      const int t = tb + ((threadIdx.x & 31) >> 3);
      route_tokens8<4 * NSLOT>(logits, t, t < T, E, k, score_fn, renorm, G, g_keep, group_score, rho, topk_idx,
                               topk_w, st);
      return;
    }
  }
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  float x[NSLOT];
  load_logits<NSLOT>(logits, t, E, x);
  route_token<NSLOT>(x, t, E, k, score_fn, renorm, G, g_keep, group_score, rho, topk_idx, topk_w,
                     s_score + (size_t)warp * E, st);
}

// S2 pass 1: per block of kScanChunk tokens, the count of entries per expert.
// Out-of-range ids are reported and counted for expert 0 (keeps every later index in
// bounds; the map is then garbage and the status word says so).
__global__ void __launch_bounds__(kScanChunk) scan_count_kernel(
    const int32_t* __restrict__ topk_idx, int T, int k, int E, int32_t* __restrict__ blockcnt,
    DeviceStatus* st) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kScanChunk + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[(int64_t)t * k + j];
      if (e < 0 || e >= E) { set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t); e = 0; }
      atomicAdd(&hist[e], 1);  // a count: the order of the adds does not show
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blockcnt[(int64_t)blockIdx.x * E + e] = hist[e];
}

// S2 pass 2 (one block): counts, offsets (exclusive scan over experts) and, in place of
// each block's count, the first row that block's entries of expert e take. Each expert's
// NB block counts are split into P contiguous shares, one per thread (P consecutive lanes),
// so the dependent chains over the blocks are P times shorter; s_off holds the experts'
// totals [E], their exclusive offsets [E] and the shares' sums [E * P].
__global__ void __launch_bounds__(1024) scan_offsets_kernel(int E, int NB, int P, int32_t* __restrict__ blockcnt,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  extern __shared__ int32_t s_off[];
  int32_t* tot_s = s_off;
  int32_t* excl_s = s_off + E;
  int32_t* part_s = s_off + 2 * E;
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (NB + P - 1) / P;  // blocks per share
  // shares and expert totals (the loop bound is the same for every thread, so the lane
  // groups are complete at every shuffle)
  for (int i0 = 0; i0 < E * P; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const int e = i / P, q = i - e * P;
    int32_t part = 0;
    if (e < E) {
      const int b1 = min(NB, (q + 1) * per);
      for (int b = q * per; b < b1; ++b) part += blockcnt[(int64_t)b * E + e];
      part_s[i] = part;
    }
    int32_t tot = part;
    for (int off = 1; off < P; off <<= 1) tot += __shfl_xor_sync(kFull, tot, off);
    if (e < E && q == 0) tot_s[e] = tot;
  }
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int32_t tot = e < E ? tot_s[e] : 0;
    int32_t inc = tot;  // inclusive warp scan
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(kFull, inc, off);
      if (lane >= off) inc += o;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      const int nw = blockDim.x >> 5;
      int32_t wv = lane < nw ? warp_tot[lane] : 0;
      int32_t wi = wv;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int32_t o = __shfl_up_sync(kFull, wi, off);
        if (lane >= off) wi += o;
      }
      if (lane < nw) warp_tot[lane] = wi - wv;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int32_t excl = carry + warp_tot[warp] + inc - tot;
    if (e < E) {
      counts[e] = tot;
      offsets[e] = excl;
      excl_s[e] = excl;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = excl + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[E] = carry;
  // each share's blocks get their first rows: the expert's offset plus the earlier shares
  for (int i0 = 0; i0 < E * P; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const int e = i / P, q = i - e * P;
    if (e < E) {
      int32_t run = excl_s[e];
      for (int qq = 0; qq < q; ++qq) run += part_s[e * P + qq];
      const int b1 = min(NB, (q + 1) * per);
      for (int b = q * per; b < b1; ++b) {
        const int32_t c = blockcnt[(int64_t)b * E + e];
        blockcnt[(int64_t)b * E + e] = run;
        run += c;
      }
    }
  }
}

// S2 pass 3: one warp per block of kScanChunk tokens walks them in ascending order, 32 at
// a time. For each expert e, bit l of mask[e] says that lane l's token chose e; the rank of
// that token among the 32 is the number of lower set bits, which keeps rows of an expert
// in ascending token order with no atomics whose order could show.
__global__ void __launch_bounds__(32) scan_assign_kernel(
    const int32_t* __restrict__ topk_idx, int T, int k, int E, const int32_t* __restrict__ base,
    int32_t* __restrict__ row_token, int32_t* __restrict__ tok_row, DeviceStatus* st) {
  extern __shared__ int32_t smem[];
  int32_t* counter = smem;
  uint32_t* mask = reinterpret_cast<uint32_t*>(smem + E);
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) {
    counter[e] = base[(int64_t)blockIdx.x * E + e];
    mask[e] = 0;
  }
  __syncwarp();
  const uint32_t below = (1u << lane) - 1u;
  for (int sub = 0; sub < kScanChunk; sub += 32) {
    const int t = blockIdx.x * kScanChunk + sub + lane;
    const bool valid = t < T;
    const int32_t* ids = topk_idx + (int64_t)t * k;
    if (valid)
      for (int j = 0; j < k; ++j) {
        int e = ids[j];
        if (e < 0 || e >= E) e = 0;
        const uint32_t old = atomicOr(&mask[e], 1u << lane);
        if (old >> lane & 1) set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);  // repeated id
      }
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        int e = ids[j];
        if (e < 0 || e >= E) e = 0;
        const int32_t r = counter[e] + __popc(mask[e] & below);
        row_token[r] = t;
        tok_row[(int64_t)t * k + j] = r;
      }
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        int e = ids[j];
        if (e < 0 || e >= E) e = 0;
        const uint32_t m = mask[e];
        if (m && 31 - __clz(m) == lane) {  // the highest lane closes expert e's batch
          counter[e] += __popc(m);
          mask[e] = 0;
        }
      }
    __syncwarp();
  }
}

// S2 for small batches (T <= kScanSmallT): the three passes above in one launch of one
// 1024-thread block. The counts come from shared-memory atomics, the offsets from one
// block-wide scan over the experts (E <= 512), and warp 0 walks the tokens in ascending
// order 32 at a time with the same lane-mask ranks as scan_assign_kernel, so the map is the
// same bit for bit. Shared memory: hist [E], counter [E], mask [E].
constexpr int kScanSmallT = 512;

__global__ void __launch_bounds__(1024) scan_small_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int E,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ row_token,
                                                          int32_t* __restrict__ tok_row, DeviceStatus* st) {
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;
  int32_t* counter = sm + E;
  uint32_t* mask = reinterpret_cast<uint32_t*>(sm + 2 * E);
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    hist[e] = 0;
    mask[e] = 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    int e = topk_idx[i];
    if (e < 0 || e >= E) { set_status(st, MOE_ERR_DEVICE_BAD_INPUT, i / k); e = 0; }
    atomicAdd(&hist[e], 1);  // a count: the order of the adds does not show
  }
  __syncthreads();
  // exclusive scan over the experts (one element per thread, E <= 512 < blockDim)
  const int e = threadIdx.x;
  const int32_t tot = e < E ? hist[e] : 0;
  int32_t inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int32_t wv = warp_tot[lane];
    int32_t wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(kFull, wi, off);
      if (lane >= off) wi += o;
    }
    warp_tot[lane] = wi - wv;
  }
  __syncthreads();
  const int32_t excl = warp_tot[warp] + inc - tot;
  if (e < E) {
    counts[e] = tot;
    offsets[e] = excl;
    counter[e] = excl;
  }
  if (e == E - 1) offsets[E] = excl + tot;
  __syncthreads();
  if (warp != 0) return;
  const uint32_t below = (1u << lane) - 1u;
  for (int t0 = 0; t0 < T; t0 += 32) {
    const int t = t0 + lane;
    const bool valid = t < T;
    const int32_t* ids = topk_idx + (int64_t)t * k;
    if (valid)
      for (int j = 0; j < k; ++j) {
        int ej = ids[j];
        if (ej < 0 || ej >= E) ej = 0;
        const uint32_t old = atomicOr(&mask[ej], 1u << lane);
        if (old >> lane & 1) set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);  // repeated id
      }
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        int ej = ids[j];
        if (ej < 0 || ej >= E) ej = 0;
        const int32_t r = counter[ej] + __popc(mask[ej] & below);
        row_token[r] = t;
        tok_row[(int64_t)t * k + j] = r;
      }
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        int ej = ids[j];
        if (ej < 0 || ej >= E) ej = 0;
        const uint32_t m = mask[ej];
        if (m && 31 - __clz(m) == lane) {  // the highest lane closes expert ej's batch
          counter[ej] += __popc(m);
          mask[ej] = 0;
        }
      }
    __syncwarp();
  }
}

// S1 + S2 in one cooperative launch (every block resident at once):
//   1. block b takes the contiguous chunk of tokens [b C, (b + 1) C) (C = ceil(T / grid)),
//      and warp w the contiguous part [bC + w W, bC + (w + 1) W) of it (W = ceil(C / warps)).
//      Each token is routed by route_token (the same ids and weights, bit for bit, as
//      route_topk_kernel), and each warp counts its part's entries per expert;
//   2. the block's counts (the sum over its warps) are published ([grid][E] in the
//      workspace), then a grid barrier;
//   3. every block reads all blocks' counts: the totals give counts and offsets (block 0
//      writes them), the blocks before it give its chunk's first row per expert, and a
//      prefix over its warps gives each warp's first row per expert. Every warp then walks
//      its own tokens in ascending order, 32 at a time, with the lane-mask ranks of
//      scan_assign_kernel. The map is the stable order by expert, then token, as before.
// The barrier is a sense-reversing one in the workspace head (counter, flag); its waits are
// bounded, and a block that gives up sets MOE_ERR_TIMEOUT and writes no map entries.
constexpr int kFusedWarps = 16;
constexpr int kFusedMaxBlocks = kFusedMaxRouteBlocks;
// Above this many counts ([grid][E]) the totals take the two-level form in phase 3.
constexpr int64_t kFusedOneLevelMax = 8192;

// The barrier's two words, each on its own 128-byte line: the arrival counter, then the flag
// the last arrival flips.
constexpr int kBarLine = 32;
static_assert(2 * kBarLine * 4 + 128 <= kWsHead, "barrier words fit the workspace head");

__device__ __forceinline__ bool fused_grid_barrier(uint32_t* bar, uint32_t nblocks, uint64_t timeout_ns,
                                                   DeviceStatus* st) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile uint32_t* flag = bar + kBarLine;
    const uint32_t f0 = *flag;  // read before arriving: the last arrival flips it
    __threadfence();            // this block's results are visible before its arrival
    const uint32_t arrived = atomicAdd(&bar[0], 1u);
    int ok = 1;
    if (arrived == nblocks - 1) {
      atomicExch(&bar[0], 0u);  // ready for the next barrier
      __threadfence();
      atomicExch(const_cast<uint32_t*>(flag), f0 ^ 1u);
    } else {
      const uint64_t t0 = tc::globaltimer_ns();
      while (*flag == f0) {
        if (tc::globaltimer_ns() - t0 > timeout_ns) {
          set_status(st, MOE_ERR_TIMEOUT, -1);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

template <int NSLOT, bool AUX>
__global__ void __launch_bounds__(32 * kFusedWarps, NSLOT >= 16 ? 1 : 2) route_fused_kernel(
    const float* __restrict__ logits, int T, int E, int k, int score_fn, int renorm, int G, int g_keep,
    int group_score, float rho, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
    int32_t* __restrict__ tok_row, int32_t* __restrict__ blockcnt, uint32_t* bar, uint64_t timeout_ns,
    DeviceStatus* st, uint64_t* __restrict__ auxp, float aux_alpha, float* __restrict__ aux_loss, int sub8) {
  extern __shared__ int32_t fsm[];
  // shared memory (fused_smem_ints on the host gives the same size):
  int32_t* wcnt = fsm;                                                  // [warps][E] counts, then rows
  uint32_t* mask = reinterpret_cast<uint32_t*>(fsm + kFusedWarps * E);  // [warps][E] lane masks
  int32_t* tot_s = fsm + 2 * kFusedWarps * E;                           // [E] totals
  int32_t* base = tot_s + E;                                            // [E] the chunk's first rows
  float* s_score = reinterpret_cast<float*>(base + E);                  // [warps][E] (group scores)
  const bool group_smem = G > 1 && g_keep < G && E != 32 * G;           // route_token's smem path
  unsigned long long* asum = reinterpret_cast<unsigned long long*>(     // [E] the chunk's aux sums
      fsm + ((2 * kFusedWarps * E + 2 * E + (group_smem ? kFusedWarps * E : 0) + 1) & ~1));
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = (T + (int)gridDim.x - 1) / (int)gridDim.x;
  const int t0 = (int)blockIdx.x * C, t1 = min(T, t0 + C);
  // a warp's part: with four tokens a warp, a multiple of 4 tokens
  const int W = sub8 ? 4 * ((C + 4 * kFusedWarps - 1) / (4 * kFusedWarps)) : (C + kFusedWarps - 1) / kFusedWarps;
  const int w0 = min(t1, t0 + warp * W), w1 = min(t1, w0 + W);
  for (int i = threadIdx.x; i < kFusedWarps * E; i += blockDim.x) {
    wcnt[i] = 0;
    mask[i] = 0;
  }
  if constexpr (AUX)
    for (int e = threadIdx.x; e < E; e += blockDim.x) asum[e] = 0;
  __syncthreads();
  // ---- 1. route the warp's tokens; count their entries per expert (and, with auxp, add up
  // their fixed-point probabilities for the auxiliary loss)
  int32_t* my_cnt = wcnt + warp * E;
  uint64_t aacc[NSLOT];
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) aacc[s] = 0;
  bool routed = false;
  if constexpr (NSLOT == 2 || NSLOT == 4 || NSLOT == 8) {
    if (sub8) {  // four tokens a warp, E = 32 NSLOT
      routed = true;
      for (int tb = w0; tb < w1; tb += 4) {
        const int t = tb + (lane >> 3);
        const bool active = t < w1;
        int my = route_tokens8<4 * NSLOT>(logits, t, active, E, k, score_fn, renorm, G, g_keep, group_score, rho,
                                          topk_idx, topk_w, st);
        if (active && (lane & 7) < k) {
          if (my < 0 || my >= E) { set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t); my = 0; }  // as the scan passes
          atomicAdd(&my_cnt[my], 1);
        }
        if constexpr (AUX) {
          for (int u = 0; u < 4 && tb + u < w1; ++u) {
            float x[NSLOT];
            load_logits<NSLOT>(logits, tb + u, E, x);
            aux_token_fixed<NSLOT>(x, E, score_fn, aacc);
          }
        }
      }
    }
  }
  float xn[NSLOT];  // the next token's logits, loaded while this one is routed
  if (!routed && w0 < w1) load_logits<NSLOT>(logits, w0, E, xn);
  for (int t = w0; t < w1 && !routed; ++t) {
    float x[NSLOT];
#pragma unroll
    for (int s = 0; s < NSLOT; ++s) x[s] = xn[s];
    if (t + 1 < w1) load_logits<NSLOT>(logits, t + 1, E, xn);
    int my = route_token<NSLOT>(x, t, E, k, score_fn, renorm, G, g_keep, group_score, rho, topk_idx, topk_w,
                                s_score + (size_t)warp * E, st);
    if (lane < k) {
      if (my < 0 || my >= E) { set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t); my = 0; }  // as the scan passes
      atomicAdd(&my_cnt[my], 1);
    }
    if constexpr (AUX) aux_token_fixed<NSLOT>(x, E, score_fn, aacc);
  }
  if constexpr (AUX) {
#pragma unroll
    for (int s = 0; s < NSLOT; ++s)
      if (aacc[s]) atomicAdd(&asum[s * 32 + lane], (unsigned long long)aacc[s]);  // integers: any order
  }
  __syncthreads();
  // the counts as [grid][E] (one level), or as [E][grid] (two levels: each expert's column
  // contiguous for the warp that scans it); the aux sums likewise
  const int nb = (int)gridDim.x, me = (int)blockIdx.x;
  const bool two_level = (int64_t)nb * E > kFusedOneLevelMax;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t c = 0;
#pragma unroll
    for (int w = 0; w < kFusedWarps; ++w) c += wcnt[w * E + e];
    const int64_t at = two_level ? (int64_t)e * nb + me : (int64_t)me * E + e;
    blockcnt[at] = c;
    if constexpr (AUX) auxp[at] = asum[e];
  }
  // A block whose barrier wait ran out leaves the map in bounds for the launches that read
  // it: no routed rows, and its chunk's entries pointing at row 0 (the status word reports
  // the failure).
  auto give_up = [&]() {
    for (int i = t0 * k + (int)threadIdx.x; i < t1 * k; i += blockDim.x) tok_row[i] = 0;
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        offsets[i] = 0;
        if (i < E) counts[i] = 0;
      }
  };
  // ---- 2. every block's counts are published
  if (!fused_grid_barrier(bar, gridDim.x, timeout_ns, st)) {
    give_up();
    return;
  }
  // ---- 3. totals and this chunk's first row per expert: the sum over all blocks' counts,
  // and over the blocks before this one (block 0 also adds up the aux sums).
  if (two_level) {
    // Two levels, so that the counts are read about once rather than once per block:
    // (a) a warp per expert column (block c % grid, warp c / grid) turns it, in place, into
    // the exclusive prefix over the blocks, and writes the column's total to counts (and its
    // aux sum to the column's first slot); (b) after a second barrier each block reads its
    // own prefixes and the totals.
    for (int ex = warp * nb + me; ex < E; ex += nb * kFusedWarps) {
      int32_t* col = blockcnt + (int64_t)ex * nb;
      int32_t cv[kFusedMaxBlocks / 32];
      int32_t sum = 0;  // over the blocks of the passes before
      unsigned long long sa = 0;
#pragma unroll
      for (int i = 0; i < kFusedMaxBlocks / 32; ++i) {  // block i * 32 + lane: coalesced
        const int bb = i * 32 + lane;
        cv[i] = bb < nb ? __ldcg(col + bb) : 0;
        if constexpr (AUX)
          if (bb < nb) sa += __ldcg(reinterpret_cast<const unsigned long long*>(auxp) + (int64_t)ex * nb + bb);
      }
#pragma unroll
      for (int i = 0; i < kFusedMaxBlocks / 32; ++i) {
        if (i * 32 >= nb) break;
        int32_t inc = cv[i];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int32_t o = __shfl_up_sync(kFull, inc, off);
          if (lane >= off) inc += o;
        }
        const int bb = i * 32 + lane;
        if (bb < nb) col[bb] = sum + inc - cv[i];
        sum += __shfl_sync(kFull, inc, 31);
      }
      if (lane == 0) counts[ex] = sum;
      if constexpr (AUX) {
#pragma unroll
        for (int off = 16; off; off >>= 1) sa += __shfl_xor_sync(kFull, sa, off);
        if (lane == 0) auxp[(int64_t)ex * nb] = sa;
      }
    }
    if (!fused_grid_barrier(bar, gridDim.x, timeout_ns, st)) {
      give_up();
      return;
    }
    unsigned __int128 v128 = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int32_t c = __ldcg(counts + e);
      tot_s[e] = c;
      base[e] = __ldcg(blockcnt + (int64_t)e * nb + me);
      if (AUX && me == 0) v128 += (unsigned __int128)(uint32_t)c * (uint64_t)__ldcg(auxp + (int64_t)e * nb);
    }
    if constexpr (AUX) {
      __shared__ unsigned __int128 red2[32];
      if (me == 0) {
        const unsigned __int128 v = block_sum_u128(v128, red2);
        if (threadIdx.x == 0) *aux_loss = aux_loss_from(v, aux_alpha, E, T, k);
      }
    }
    __syncthreads();
  } else {
    const bool aux_here = AUX && blockIdx.x == 0;
    unsigned __int128 v128 = 0;
    if ((E & 3) == 0 && !aux_here) {
      // P consecutive threads (a power of two) per 4 experts, 16-byte loads of every P-th
      // block's counts, then a sum over the P lanes (block 0 of the aux instance, which also
      // adds up the aux sums, takes the per-expert loop below: measured faster for it)
      const int NQ = E >> 2;
      int P = 1;
      while (P < 32 && 2 * P * NQ <= (int)blockDim.x) P *= 2;
      const int q = threadIdx.x / P, ph = threadIdx.x % P;
      int32_t tt[4] = {0, 0, 0, 0}, bf[4] = {0, 0, 0, 0};
      if (q < NQ) {
#pragma unroll 8
        for (int bb = ph; bb < nb; bb += P) {
          const int4 c = __ldcg(reinterpret_cast<const int4*>(blockcnt + (int64_t)bb * E) + q);
          tt[0] += c.x; tt[1] += c.y; tt[2] += c.z; tt[3] += c.w;
          if (bb < me) { bf[0] += c.x; bf[1] += c.y; bf[2] += c.z; bf[3] += c.w; }
        }
      }
      for (int off = 1; off < P; off <<= 1) {  // within aligned groups of P lanes
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tt[i] += __shfl_xor_sync(kFull, tt[i], off);
          bf[i] += __shfl_xor_sync(kFull, bf[i], off);
        }
      }
      if (q < NQ && ph == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          tot_s[4 * q + i] = tt[i];
          base[4 * q + i] = bf[i];
        }
      }
    } else {
      // P consecutive threads (a power of two) per expert, each adding every P-th block's count
      int P = 1;
      while (P < 32 && 2 * P * E <= (int)blockDim.x) P *= 2;
      const int ex = threadIdx.x / P, q = threadIdx.x % P;
      int32_t tot = 0, before = 0;
      unsigned long long S = 0;
      if (ex < E) {
#pragma unroll 4
        for (int bb = q; bb < nb; bb += P) {
          const int32_t c = __ldcg(blockcnt + (int64_t)bb * E + ex);
          tot += c;
          if (bb < me) before += c;
          if (aux_here) S += __ldcg(reinterpret_cast<const unsigned long long*>(auxp) + (int64_t)bb * E + ex);
        }
      }
      for (int off = 1; off < P; off <<= 1) {
        tot += __shfl_xor_sync(kFull, tot, off);
        before += __shfl_xor_sync(kFull, before, off);
        if (aux_here) S += __shfl_xor_sync(kFull, S, off);
      }
      if (ex < E && q == 0) {
        tot_s[ex] = tot;
        base[ex] = before;
        if (aux_here) v128 = (unsigned __int128)(uint32_t)tot * (uint64_t)S;
      }
    }
    if constexpr (AUX) {
      __shared__ unsigned __int128 red128[32];
      if (aux_here) {
        const unsigned __int128 v = block_sum_u128(v128, red128);
        if (threadIdx.x == 0) *aux_loss = aux_loss_from(v, aux_alpha, E, T, k);
      }
    }
    __syncthreads();
  }
  // offsets: an exclusive scan of the totals over the experts (E <= blockDim)
  const int e = threadIdx.x;
  const int32_t tot = e < E ? tot_s[e] : 0;
  int32_t inc = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int32_t wv = lane < kFusedWarps ? warp_tot[lane] : 0;
    int32_t wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(kFull, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kFusedWarps) warp_tot[lane] = wi - wv;
  }
  __syncthreads();
  const int32_t excl = warp_tot[warp] + inc - tot;
  if (e < E) {
    int32_t run = excl + base[e];  // the chunk's first row for expert e, then each warp's
#pragma unroll
    for (int w = 0; w < kFusedWarps; ++w) {
      const int32_t c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    if (blockIdx.x == 0) {
      counts[e] = tot;
      offsets[e] = excl;
      if (e == E - 1) offsets[E] = excl + tot;
    }
  }
  __syncthreads();
  // ---- the warp's rows, its tokens in ascending order (their ids were written by this warp)
  int32_t* wrow = wcnt + warp * E;
  uint32_t* wmask = mask + warp * E;
  const int64_t R = (int64_t)T * k;
  const uint32_t below = (1u << lane) - 1u;
  for (int tb = w0; tb < w1; tb += 32) {
    const int t = tb + lane;
    const bool valid = t < w1;
    const int32_t* ids = topk_idx + (int64_t)t * k;
    auto id_of = [&](int j) {
      const int ej = ids[j];
      return (ej < 0 || ej >= E) ? 0 : ej;  // counted for expert 0 above (status set)
    };
    if (valid)
      for (int j = 0; j < k; ++j) atomicOr(&wmask[id_of(j)], 1u << lane);
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        const int ej = id_of(j);
        const int64_t r = wrow[ej] + __popc(wmask[ej] & below);
        if (r >= 0 && r < R) {
          row_token[r] = t;
          tok_row[(int64_t)t * k + j] = (int32_t)r;
        } else {
          set_status(st, MOE_ERR_DEVICE_BAD_INPUT, t);
        }
      }
    __syncwarp();
    if (valid)
      for (int j = 0; j < k; ++j) {
        const int ej = id_of(j);
        const uint32_t m = wmask[ej];
        if (m && 31 - __clz(m) == lane) {  // the highest lane closes expert ej's batch
          wrow[ej] += __popc(m);
          wmask[ej] = 0;
        }
      }
    __syncwarp();
  }
}

// S0 for small expert counts (E <= EP <= 32): one 256-thread block per TB tokens; the
// threads split the hidden dimension (16-byte chunks c = tid, tid + 256, ...), each keeping
// TB x E partial dot products, then a warp reduction and a cross-warp sum through smem.
// Splitting H over the block keeps many independent loads in flight per SM, which is what
// this memory-bound pass needs. fp32 accumulation.
template <int EP, int TB, bool BF16>
__global__ void __launch_bounds__(256) router_small_kernel(const void* __restrict__ x_, const void* __restrict__ w_,
                                                           const float* __restrict__ bias, int T, int H, int E,
                                                           float* __restrict__ logits) {
  __shared__ float part[8][TB][EP];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int EPC = BF16 ? 8 : 4;  // elements per 16-byte chunk
  const int nchunk = H / EPC;
  const int t0 = blockIdx.x * TB;
  float acc[TB][EP];
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[i][e] = 0.0f;
  for (int c = threadIdx.x; c < nchunk; c += 256) {
    float xf[TB][EPC];
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      const int t = min(t0 + i, T - 1);  // a short last block repeats a row; not stored
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x_) + (int64_t)t * nchunk + c);
      if (BF16) {
        const uint32_t u[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) { xf[i][2 * q] = __uint_as_float(u[q] << 16); xf[i][2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u); }
      } else {
        xf[i][0] = __uint_as_float(xv.x); xf[i][1] = __uint_as_float(xv.y);
        xf[i][2] = __uint_as_float(xv.z); xf[i][3] = __uint_as_float(xv.w);
      }
    }
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      if (e < E) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(w_) + (int64_t)e * nchunk + c);
        float wf[EPC];
        if (BF16) {
          const uint32_t u[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) { wf[2 * q] = __uint_as_float(u[q] << 16); wf[2 * q + 1] = __uint_as_float(u[q] & 0xffff0000u); }
        } else {
          wf[0] = __uint_as_float(wv.x); wf[1] = __uint_as_float(wv.y);
          wf[2] = __uint_as_float(wv.z); wf[3] = __uint_as_float(wv.w);
        }
#pragma unroll
        for (int i = 0; i < TB; ++i)
#pragma unroll
          for (int q = 0; q < EPC; ++q) acc[i][e] = __fmaf_rn(xf[i][q], wf[q], acc[i][e]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      float v = acc[i][e];
#pragma unroll
      for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      if (lane == 0) part[warp][i][e] = v;
    }
  __syncthreads();
  if (threadIdx.x < TB * EP) {
    const int i = threadIdx.x / EP, e = threadIdx.x % EP;
    if (e < E && t0 + i < T) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += part[w][i][e];
      logits[(int64_t)(t0 + i) * E + e] = bias ? v + bias[e] : v;
    }
  }
}

// S0 on the tensor cores for bf16 x with E <= 32 experts (HBM-bound: x is read once):
// mma.sync m16n8k16 (bf16 x bf16 -> fp32). A block takes 16 tokens; its NW warps split the
// row's 32-wide K steps into NW contiguous ranges. In a step, thread (g = lane / 4,
// q = lane % 4) loads 16 contiguous bytes (8 bf16 at k0 + 8 q) of token rows g and g + 8
// and of expert row nt * 8 + g for each of the NT 8-expert tiles. The step's two MMAs take
// those as a fixed permutation of the 32 K positions (the same for x and W, so each product
// x[t, k] W[e, k] is formed once): the first MMA's K slots 2q, 2q + 1 hold k0 + 8q + {0, 1}
// and slots 2q + 8, 2q + 9 hold k0 + 8q + {2, 3}; the second MMA the same with + 4. A warp
// loads U steps into registers before it issues their MMAs, so that U steps of loads are in
// flight per warp: the kernel is bound by how many bytes of x are in flight, not by the MMAs.
// The warps' fp32 partial logits are added in warp order through shared memory, then the
// bias.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NW warps a block: 8 for one 8-expert tile, so that two 256-thread blocks fit an SM's
// registers and the whole grid is resident at once; 16 for wider E, whose fewer steps in
// flight per warp are made up by more warps.
template <int NT, int NW>
__global__ void __launch_bounds__(32 * NW) router_hmma_kernel(const uint4* __restrict__ x,
                                                                         const uint4* __restrict__ w,
                                                                         const float* __restrict__ bias, int T, int H,
                                                                         int E, float* __restrict__ logits) {
  constexpr int U = NT == 1 ? 8 : NT == 2 ? 4 : 2;  // steps in flight per warp (registers: U (2 + NT) uint4)
  __shared__ float red[NW][16][8 * NT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int t0 = blockIdx.x * 16;
  const int row_chunks = H / 8;  // 16-byte chunks of a row
  const int ta = min(t0 + g, T - 1), tb = min(t0 + g + 8, T - 1);  // past T: a repeated row, not stored
  const uint4* xa = x + (int64_t)ta * row_chunks + q;
  const uint4* xb = x + (int64_t)tb * row_chunks + q;
  const uint4* wr[NT];
  bool wok[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int e = nt * 8 + g;
    wok[nt] = e < E;
    wr[nt] = w + (int64_t)(wok[nt] ? e : 0) * row_chunks + q;
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
  const int S = H / 32;                                    // 32-wide K steps of a row
  const int per = (S + NW - 1) / NW;                      // steps of a warp
  const int s_end = min(S, (warp + 1) * per);
  for (int sb = warp * per; sb < s_end; sb += U) {
    uint4 va[U], vb[U], vw[U][NT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (sb + u < s_end) {
        const int c = (sb + u) * 4;  // 4 chunks a step
        va[u] = __ldg(xa + c);
        vb[u] = __ldg(xb + c);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) vw[u][nt] = wok[nt] ? __ldg(wr[nt] + c) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (sb + u < s_end) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_bf16_16816(acc[nt], va[u].x, vb[u].x, va[u].y, vb[u].y, vw[u][nt].x, vw[u][nt].y);
          mma_bf16_16816(acc[nt], va[u].z, vb[u].z, va[u].w, vb[u].w, vw[u][nt].z, vw[u][nt].w);
        }
      }
    }
  }
  // D fragment: (token g, expert nt * 8 + 2q + {0, 1}) and (token g + 8, the same experts)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][g][nt * 8 + 2 * q] = acc[nt][0];
    red[warp][g][nt * 8 + 2 * q + 1] = acc[nt][1];
    red[warp][g + 8][nt * 8 + 2 * q] = acc[nt][2];
    red[warp][g + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * 8 * NT; i += blockDim.x) {
    const int tl = i / (8 * NT), e = i % (8 * NT);
    const int t = t0 + tl;
    if (t < T && e < E) {
      float v = 0.0f;
#pragma unroll
      for (int wp = 0; wp < NW; ++wp) v += red[wp][tl][e];
      logits[(int64_t)t * E + e] = bias ? v + bias[e] : v;
    }
  }
}

// Auxiliary load-balancing loss, pass 1: per block of 128 tokens (8 warps x 16 tokens), the
// sum over its tokens of each expert's fixed-point probability (aux_token_fixed).
template <int NSLOT>
__global__ void __launch_bounds__(256) aux_pbar_kernel(const float* __restrict__ logits, int T, int E,
                                                       int score_fn, uint64_t* __restrict__ part) {
  __shared__ unsigned long long wsum[NSLOT * 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < NSLOT * 32; e += blockDim.x) wsum[e] = 0;
  __syncthreads();
  uint64_t acc[NSLOT];
#pragma unroll
  for (int s = 0; s < NSLOT; ++s) acc[s] = 0;
  for (int i = 0; i < 16; ++i) {
    const int t = blockIdx.x * 128 + warp * 16 + i;
    if (t >= T) break;
    float x[NSLOT];
    load_logits<NSLOT>(logits, t, E, x);
    aux_token_fixed<NSLOT>(x, E, score_fn, acc);
  }
#pragma unroll
  for (int s = 0; s < NSLOT; ++s)
    if (acc[s]) atomicAdd(&wsum[s * 32 + lane], (unsigned long long)acc[s]);  // integers: any order
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) part[(int64_t)blockIdx.x * E + e] = wsum[e];
}

// Pass 2 (one block): S_e = the sum over blocks, then the loss from the exact
// V = sum_e counts[e] * S_e.
__global__ void __launch_bounds__(1024) aux_loss_kernel(const uint64_t* __restrict__ part, int NB, int E,
                                                        const int32_t* __restrict__ counts, int T, int k,
                                                        float alpha, float* __restrict__ loss) {
  __shared__ unsigned __int128 red[32];
  unsigned __int128 v = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    uint64_t se = 0;
    for (int b = 0; b < NB; ++b) se += part[(int64_t)b * E + e];
    v += (unsigned __int128)(uint32_t)max(counts[e], 0) * se;
  }
  v = block_sum_u128(v, red);
  if (threadIdx.x == 0) *loss = aux_loss_from(v, alpha, E, T, k);
}

}  // namespace

cudaError_t launch_aux_loss(const moe_config_t& c, const float* logits, const int32_t* counts, float alpha,
                            float* loss, uint64_t* part, cudaStream_t s) {
  const int NB = scan_blocks(c);
  const int nslot = (int)ceil_div(c.E, 32);
  if (NB > 0) {
#define MOE_AUX(NS) \
  if (nslot <= NS) aux_pbar_kernel<NS><<<NB, 256, 0, s>>>(logits, c.T, c.E, c.score_fn, part); else
    MOE_AUX(1) MOE_AUX(2) MOE_AUX(4) MOE_AUX(8) MOE_AUX(16) return cudaErrorInvalidValue;
#undef MOE_AUX
  }
  aux_loss_kernel<<<1, 1024, 0, s>>>(part, NB, c.E, counts, c.T > 0 ? c.T : 1, c.k, alpha, loss);
  return cudaGetLastError();
}

bool router_small_supported(const moe_config_t& c) { return c.E <= 32; }

cudaError_t launch_router_small(const moe_config_t& c, const void* x, const void* w, const float* bias,
                                float* logits, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const bool bf = c.act_dtype == MOE_DTYPE_BF16;
  // bf16 rows of a multiple of 256: the tensor-core form, 16 tokens a block
  if (bf && c.H % 256 == 0) {
    const unsigned blocks = (unsigned)ceil_div(c.T, 16);
    const uint4* xv = static_cast<const uint4*>(x);
    const uint4* wv = static_cast<const uint4*>(w);
#define MOE_RH(NT) \
  if (c.E <= 8 * NT) { \
    constexpr int NW = NT == 1 ? 8 : 16; \
    router_hmma_kernel<NT, NW><<<blocks, 32 * NW, 0, s>>>(xv, wv, bias, c.T, c.H, c.E, logits); \
    return cudaGetLastError(); \
  }
    MOE_RH(1) MOE_RH(2) MOE_RH(3) MOE_RH(4)
#undef MOE_RH
  }
#define MOE_RS(EP, TB)                                                                                \
  if (c.E <= EP) {                                                                                  \
    const unsigned blocks = (unsigned)ceil_div(c.T, TB);                                            \
    if (bf) router_small_kernel<EP, TB, true><<<blocks, 256, 0, s>>>(x, w, bias, c.T, c.H, c.E, logits); \
    else router_small_kernel<EP, TB, false><<<blocks, 256, 0, s>>>(x, w, bias, c.T, c.H, c.E, logits);   \
    return cudaGetLastError();                                                                      \
  }
  MOE_RS(8, 2)
  MOE_RS(16, 2)
  MOE_RS(32, 1)
#undef MOE_RS
  return cudaErrorInvalidValue;
}

namespace {
// Four tokens a warp where the shape allows it and the logits rows are 16-byte aligned
// (the routine reads them as float4); every launch that routes a configuration makes the
// same choice, so the routing kernels give the same bits.
int route_sub8_for(const moe_config_t& c, const float* logits) {
  return route_sub8(c.E, c.k, c.n_groups, c.topk_groups) && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
}

}  // namespace

cudaError_t launch_route_topk(const moe_config_t& c, const float* logits, int32_t* topk_idx,
                              float* topk_w, DeviceStatus* st, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  const int warps = 8;
  const int sub8 = route_sub8_for(c, logits);  // four tokens a warp
  const dim3 grid((unsigned)ceil_div(c.T, sub8 ? 4 * warps : warps)), block(warps * 32);
  const bool grouped = c.n_groups > 1 && c.topk_groups < c.n_groups;
  const size_t smem = grouped && !sub8 ? (size_t)warps * c.E * sizeof(float) : 0;
  const int nslot = (int)ceil_div(c.E, 32);
#define MOE_ROUTE_CASE(NS)                                                                  \
  if (nslot <= NS) {                                                                        \
    route_topk_kernel<NS><<<grid, block, smem, s>>>(logits, c.T, c.E, c.k, c.score_fn,      \
                                                    c.renorm, c.n_groups, c.topk_groups,    \
                                                    c.group_score, c.routed_scale, topk_idx, \
                                                    topk_w, st, sub8);                      \
    return cudaGetLastError();                                                              \
  }
  MOE_ROUTE_CASE(1)
  MOE_ROUTE_CASE(2)
  MOE_ROUTE_CASE(4)
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(16)
#undef MOE_ROUTE_CASE
  return cudaErrorInvalidValue;
}

namespace {

// The fused kernel's instance, its shared memory and its grid for a configuration.
struct FusedPlan {
  const void* kern = nullptr;      // plain routing
  const void* kern_aux = nullptr;  // routing + auxiliary loss
  size_t smem = 0, smem_aux = 0;
  int64_t grid = 0;
};

template <int NS, bool AUX>
const void* fused_kernel_ptr() { return reinterpret_cast<const void*>(&route_fused_kernel<NS, AUX>); }

template <bool AUX>
const void* fused_kernel_for(int nslot) {
  return nslot <= 1 ? fused_kernel_ptr<1, AUX>() : nslot <= 2 ? fused_kernel_ptr<2, AUX>()
       : nslot <= 4 ? fused_kernel_ptr<4, AUX>() : nslot <= 8 ? fused_kernel_ptr<8, AUX>()
       : nslot <= 16 ? fused_kernel_ptr<16, AUX>() : nullptr;
}

// Blocks per SM of one fused instance with `smem` bytes of dynamic shared memory (cached per
// instance and size); 0 on failure.
int fused_per_sm(const void* kern, size_t smem) {
  struct Entry { const void* kern; size_t smem; int per_sm; };
  static Entry cache[4] = {};
  static int next = 0;
  for (const Entry& e : cache)
    if (e.kern == kern && e.smem == smem) return e.per_sm;
  if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 32 * kFusedWarps, smem) != cudaSuccess) return 0;
  cache[next] = Entry{kern, smem, per_sm};
  next = (next + 1) % 4;
  return per_sm;
}

// The plain instance routes (moe_route); the AUX one also forms the auxiliary loss
// (moe_forward_train). Both take the same grid, sized so that either is resident at once.
FusedPlan fused_plan(const moe_config_t& c) {
  FusedPlan f;
  const int nslot = (int)ceil_div(c.E, 32);
  f.kern = fused_kernel_for<false>(nslot);
  f.kern_aux = fused_kernel_for<true>(nslot);
  if (!f.kern || !f.kern_aux) return f;
  const bool group_smem = c.n_groups > 1 && c.topk_groups < c.n_groups && c.E != 32 * c.n_groups;
  // per-warp counts and lane masks [warps][E], totals and first rows [E] ints, and the group
  // scores [warps][E] floats where route_token stages them; the AUX instance adds the aux
  // sums [E] 64-bit integers at an 8-byte boundary
  const size_t ints =
      (size_t)((2 * kFusedWarps * c.E + 2 * c.E + (group_smem ? kFusedWarps * c.E : 0) + 1) & ~1);
  f.smem = ints * sizeof(int32_t);
  f.smem_aux = f.smem + (size_t)c.E * sizeof(uint64_t);
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  const int per_sm = std::min(fused_per_sm(f.kern, f.smem), fused_per_sm(f.kern_aux, f.smem_aux));
  if (per_sm <= 0) return f;
  // every block resident at once (the grid barrier), and at most one block per 16 tokens
  f.grid = std::max<int64_t>(
      1, std::min<int64_t>(std::min<int64_t>((int64_t)per_sm * sms, kFusedMaxBlocks), ceil_div(c.T, kFusedWarps)));
  return f;
}

}  // namespace

// The fused launch where its top-k phase stays short: a warp routes its part of the block's
// chunk one token after another, at a cost per token that grows with E / 32 (the slots a
// lane holds), so the chunk times the slots is kept to at most 1024 (e.g. 108 tokens a block
// of 256 grouped experts at T = 32768). Longer chunks keep the top-k launch, one warp per
// token, and the scan passes.
bool route_fused_supported(const moe_config_t& c) {
  if (c.T <= 0 || c.E > 32 * kFusedWarps || c.k > 32) return false;
  const FusedPlan f = fused_plan(c);
  if (f.grid <= 0) return false;
  return ceil_div(c.T, f.grid) * ceil_div(c.E, 32) <= 1024;
}

cudaError_t launch_route_fused(const moe_config_t& c, const float* logits, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* tok_row,
                               int32_t* blockcnt, uint32_t* barrier, DeviceStatus* st, cudaStream_t s,
                               uint64_t* auxp, float aux_alpha, float* aux_loss) {
  if (c.T == 0) return cudaSuccess;
  const FusedPlan f = fused_plan(c);
  if (f.grid <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  const int sub8 = route_sub8_for(c, logits);
  cfg.gridDim = dim3((unsigned)f.grid);
  cfg.blockDim = dim3(32 * kFusedWarps);
  cfg.dynamicSmemBytes = auxp ? f.smem_aux : f.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint64_t timeout = 2000000000ull;
  void* args[] = {(void*)&logits,  (void*)&c.T,           (void*)&c.E,          (void*)&c.k,
                  (void*)&c.score_fn, (void*)&c.renorm,   (void*)&c.n_groups,   (void*)&c.topk_groups,
                  (void*)&c.group_score, (void*)&c.routed_scale, (void*)&topk_idx, (void*)&topk_w,
                  (void*)&counts,  (void*)&offsets,       (void*)&row_token,    (void*)&tok_row,
                  (void*)&blockcnt, (void*)&barrier,      (void*)&timeout,      (void*)&st,
                  (void*)&auxp,    (void*)&aux_alpha,     (void*)&aux_loss, (void*)&sub8};
  cudaError_t e = cudaLaunchKernelExC(&cfg, auxp ? f.kern_aux : f.kern, args);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_route_scan(const moe_config_t& c, const int32_t* topk_idx, int32_t* counts,
                              int32_t* offsets, int32_t* row_token, int32_t* tok_row,
                              int32_t* blockcnt, DeviceStatus* st, cudaStream_t s) {
  if (c.T > 0 && c.T <= kScanSmallT) {  // small batches: one launch
    scan_small_kernel<<<1, 1024, (size_t)3 * c.E * sizeof(int32_t), s>>>(topk_idx, c.T, c.k, c.E, counts, offsets,
                                                                         row_token, tok_row, st);
    return cudaGetLastError();
  }
  const int NB = scan_blocks(c);
  if (NB > 0) {
    scan_count_kernel<<<NB, kScanChunk, c.E * sizeof(int32_t), s>>>(topk_idx, c.T, c.k, c.E, blockcnt, st);
  }
  int P = 1;  // threads per expert in the offsets pass: a power of two, at most 32
  while (P < 32 && 2 * P * c.E <= 1024) P *= 2;
  scan_offsets_kernel<<<1, 1024, (size_t)(2 + P) * c.E * sizeof(int32_t), s>>>(c.E, NB, P, blockcnt, counts,
                                                                             offsets);
  if (NB > 0) {
    scan_assign_kernel<<<NB, 32, 2 * c.E * sizeof(int32_t), s>>>(topk_idx, c.T, c.k, c.E, blockcnt,
                                                                 row_token, tok_row, st);
  }
  return cudaGetLastError();
}

}  // namespace moe
