/*
 * CPU oracle for the single-GPU MoE layer forward: test infrastructure only.
 *
 * Plain, slow, obviously correct C, fp64 unless a step fixes another precision. It shares
 * no code with the CUDA library (no header, helper or table); only the tests, the smoke
 * check and the benchmark's CPU-baseline leg call it. Each function names the passage of
 * the method it follows. The pages ("Scalable Training of Mixture-of-Experts Models with
 * Megatron Core" summary, the Megatron-Core distributed-training skill card, the Piper
 * summary and the Hybrid-EP article) state WHAT the layer does but print no formula; where
 * they are silent the plainest reading is taken and named at the function.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math: the
 * routing scores below must be computed with exactly the IEEE operations written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------------------ */
/* Deterministic fp32 exp: Cody-Waite argument reduction (W. J. Cody and W. Waite,       */
/* "Software Manual for the Elementary Functions", 1980) with a two-constant split of    */
/* ln 2, a degree-7 Taylor polynomial of e^r on |r| <= ln2/2 evaluated by Horner with     */
/* fused multiply-adds, and an exact power-of-two scaling in two steps.                   */
/* Every operation is a correctly rounded IEEE fp32 operation, so any machine that        */
/* performs the same sequence gets the same bits. Used only where an fp32 value decides  */
/* an integer (the sigmoid group scores of group-limited routing).                        */
/* ------------------------------------------------------------------------------------ */
static float pow2i(int n) { /* 2^n for n in [-126, 127], exact */
  union { uint32_t u; float f; } v;
  v.u = (uint32_t)(n + 127) << 23;
  return v.f;
}

float oc_det_expf(float a) {
  if (a != a) return a;
  if (a > 88.72283935546875f) return INFINITY;
  if (a < -103.972084045410156f) return 0.0f;
  const float log2e = 1.44269502162933349609375f;      /* fp32(1/ln 2) */
  const float ln2_hi = 0.693145751953125f;              /* 0x3F317200: 16 significant bits */
  const float ln2_lo = 1.428606765330187045e-06f;       /* 0x35BFBE8E: fp32(ln2 - ln2_hi) */
  float t = a * log2e;
  float n = rintf(t);
  float r = fmaf(-n, ln2_hi, a);
  r = fmaf(-n, ln2_lo, r);
  /* e^r = sum r^i / i!, i = 0..7 */
  float p = 1.98412698412698412698e-04f;                /* 1/7! */
  p = fmaf(p, r, 1.38888888888888888889e-03f);          /* 1/6! */
  p = fmaf(p, r, 8.33333333333333333333e-03f);          /* 1/5! */
  p = fmaf(p, r, 4.16666666666666666667e-02f);          /* 1/4! */
  p = fmaf(p, r, 1.66666666666666666667e-01f);          /* 1/3! */
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n;
  int n1 = ni >> 1; /* floor(n/2); n1, n - n1 in [-75, 64] */
  int n2 = ni - n1;
  return (p * pow2i(n1)) * pow2i(n2);
}

/* s = 1 / (1 + e^-l), fp32, with the deterministic exp above. */
float oc_det_sigmoidf(float l) { return 1.0f / (1.0f + oc_det_expf(-l)); }

void oc_det_expf_array(const float* a, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oc_det_expf(a[i]);
}

/* ------------------------------------------------------------------------------------ */
/* S0: router logits. l[t,e] = sum_h x[t,h] * Wr[e,h] (+ b[e]) accumulated in fp64 from   */
/* the stored values, rounded once to fp32: the router gives every token one score per   */
/* expert (Megatron-Core summary, section "O essencial"); the synthetic router weights    */
/* are drawn N(0, 0.02^2). b is the optional per-expert additive bias of the imbalanced   */
/* workload.                                                                              */
/* ------------------------------------------------------------------------------------ */
void oc_router_logits(const float* x, const float* wr, const float* bias, int T, int H, int E,
                      float* logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += (double)x[(int64_t)t * H + h] * (double)wr[(int64_t)e * H + h];
      if (bias) s += (double)bias[e];
      logits[(int64_t)t * E + e] = (float)s;
    }
}

/* ------------------------------------------------------------------------------------ */
/* S1: top-k routing with optional group-limited selection.                               */
/* Key = fp32 logit, descending; equal keys go to the lower expert index (softmax and     */
/* sigmoid are strictly increasing, so this is the ranking by score). Group-limited       */
/* selection (DeepSeek-V3 shape: 256 experts, top-8; Hybrid-EP article results) keeps    */
/* the topk_groups groups of contiguous experts with the largest group score, ties to the */
/* lower group; group score = sum of the two largest fp32 sigmoid scores in the group     */
/* (group_score 0) or the largest (group_score 1), scores from oc_det_sigmoidf.           */
/* Weights (fp64): softmax over all experts, or over the selected ones when renorm;       */
/* sigmoid s_j, divided by the selected sum when renorm; then times routed_scale.         */
/* Returns 0, or -1 if a logit is not finite.                                             */
/* ------------------------------------------------------------------------------------ */
typedef struct { float key; int idx; } oc_kv;

static int kv_desc(const void* a, const void* b) {
  const oc_kv* p = (const oc_kv*)a;
  const oc_kv* q = (const oc_kv*)b;
  if (p->key > q->key) return -1;
  if (p->key < q->key) return 1;
  return (p->idx < q->idx) ? -1 : (p->idx > q->idx);
}

static int route_one(const float* l, int E, int k, int score_fn, int renorm, int n_groups,
                     int topk_groups, int group_score, double routed_scale, int32_t* idx_out,
                     double* w_out, float* group_scores_out) {
  for (int e = 0; e < E; ++e)
    if (!isfinite(l[e])) return -1;
  oc_kv* kv = (oc_kv*)malloc(sizeof(oc_kv) * (size_t)E);
  char* allowed = (char*)malloc((size_t)E);
  for (int e = 0; e < E; ++e) allowed[e] = 1;
  if (n_groups > 1 && topk_groups < n_groups) {
    int gs = E / n_groups;
    oc_kv* gk = (oc_kv*)malloc(sizeof(oc_kv) * (size_t)n_groups);
    float* s = (float*)malloc(sizeof(float) * (size_t)gs);
    for (int g = 0; g < n_groups; ++g) {
      for (int i = 0; i < gs; ++i) s[i] = oc_det_sigmoidf(l[g * gs + i]);
      float m1 = -INFINITY, m2 = -INFINITY; /* two largest scores */
      for (int i = 0; i < gs; ++i) {
        if (s[i] > m1) { m2 = m1; m1 = s[i]; }
        else if (s[i] > m2) m2 = s[i];
      }
      float sc = (group_score == 0 && gs >= 2) ? (m1 + m2) : m1;
      gk[g].key = sc;
      gk[g].idx = g;
      if (group_scores_out) group_scores_out[g] = sc;
    }
    qsort(gk, (size_t)n_groups, sizeof(oc_kv), kv_desc);
    for (int e = 0; e < E; ++e) allowed[e] = 0;
    for (int r = 0; r < topk_groups; ++r)
      for (int i = 0; i < gs; ++i) allowed[gk[r].idx * gs + i] = 1;
    free(s);
    free(gk);
  }
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (allowed[e]) { kv[n].key = l[e]; kv[n].idx = e; ++n; }
  qsort(kv, (size_t)n, sizeof(oc_kv), kv_desc);
  for (int j = 0; j < k; ++j) idx_out[j] = kv[j].idx;

  if (score_fn == 0) {
    double m = -INFINITY;
    for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
    double denom = 0.0;
    if (renorm) for (int j = 0; j < k; ++j) denom += exp((double)l[idx_out[j]] - m);
    else for (int e = 0; e < E; ++e) denom += exp((double)l[e] - m);
    for (int j = 0; j < k; ++j) w_out[j] = routed_scale * exp((double)l[idx_out[j]] - m) / denom;
  } else {
    double sum = 0.0, sj[1024];
    for (int j = 0; j < k; ++j) { sj[j] = 1.0 / (1.0 + exp(-(double)l[idx_out[j]])); sum += sj[j]; }
    for (int j = 0; j < k; ++j) w_out[j] = routed_scale * (renorm ? sj[j] / sum : sj[j]);
  }
  free(allowed);
  free(kv);
  return 0;
}

int oc_route(const float* logits, int T, int E, int k, int score_fn, int renorm, int n_groups,
             int topk_groups, int group_score, double routed_scale, int32_t* topk_idx,
             double* topk_w) {
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int t = 0; t < T; ++t)
    if (route_one(logits + (int64_t)t * E, E, k, score_fn, renorm, n_groups, topk_groups,
                  group_score, routed_scale, topk_idx + (int64_t)t * k, topk_w + (int64_t)t * k,
                  NULL))
      bad = 1;
  return bad ? -1 : 0;
}

/* Group scores of one token (for tests of the group step). */
int oc_group_scores(const float* l, int E, int n_groups, int group_score, float* out) {
  int gs = E / n_groups;
  float* s = (float*)malloc(sizeof(float) * (size_t)gs);
  for (int g = 0; g < n_groups; ++g) {
    for (int i = 0; i < gs; ++i) s[i] = oc_det_sigmoidf(l[g * gs + i]);
    float m1 = -INFINITY, m2 = -INFINITY;
    for (int i = 0; i < gs; ++i) {
      if (s[i] > m1) { m2 = m1; m1 = s[i]; }
      else if (s[i] > m2) m2 = s[i];
    }
    out[g] = (group_score == 0 && gs >= 2) ? (m1 + m2) : m1;
  }
  free(s);
  return 0;
}

/* ------------------------------------------------------------------------------------ */
/* S2: per-expert counts, offsets and the permutation. counts[e] = #{(t,j): idx=e};        */
/* offsets = exclusive prefix sum (offsets[E] = T*k); within expert e the rows hold the    */
/* tokens that chose e in ascending token id (the routing map of the Hybrid-EP article,  */
/* whose order the pages leave open; the stable order is the reading taken).              */
/* row_token[r] = t, tok_row[t*k+j] = r.                                                  */
/* Returns 0, or -1 if an expert id is outside [0, E).                                    */
/* ------------------------------------------------------------------------------------ */
int oc_permute(const int32_t* topk_idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
               int32_t* row_token, int32_t* tok_row) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t i = 0; i < (int64_t)T * k; ++i) {
    int e = topk_idx[i];
    if (e < 0 || e >= E) return -1;
    counts[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = topk_idx[(int64_t)t * k + j];
      int r = offsets[e] + fill[e]++;
      row_token[r] = t;
      tok_row[(int64_t)t * k + j] = r;
    }
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------------------------ */
/* S3: dispatch, xd[r] = x[row_token[r]] (the Hybrid-EP article's dispatch operator, which */
/* moves each token to the experts it was routed to). Bit copy.                           */
/* ------------------------------------------------------------------------------------ */
void oc_dispatch(const float* x, int H, const int32_t* row_token, int64_t nrows, float* xd) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r)
    memcpy(xd + r * H, x + (int64_t)row_token[r] * H, sizeof(float) * (size_t)H);
}

/* ------------------------------------------------------------------------------------ */
/* FP8 e4m3 (OCP 8-bit floating point specification, E4M3 "fn" variant): 1 sign bit,     */
/* 4 exponent bits (bias 7), 3 mantissa bits, no infinities, max finite 448, one NaN      */
/* pattern per sign (S.1111.111). Encoding rounds to nearest, ties to even, and          */
/* saturates finite values beyond 448 to +-448 ("satfinite").                             */
/* ------------------------------------------------------------------------------------ */
double oc_e4m3_decode(uint8_t c) {
  int s = c >> 7, ex = (c >> 3) & 15, m = c & 7;
  double v;
  if (ex == 15 && m == 7) return NAN;
  if (ex == 0) v = ldexp((double)m, -9);           /* subnormal: m * 2^-6 / 8 */
  else v = ldexp(8.0 + m, ex - 7 - 3);              /* (1 + m/8) * 2^(ex-7) */
  return s ? -v : v;
}

uint8_t oc_e4m3_encode(float f) {
  if (f != f) return 0x7F;
  int s = signbit(f) ? 1 : 0;
  double a = fabs((double)f);
  uint8_t code;
  if (a >= 448.0) code = 0x7E;                       /* satfinite */
  else if (a < ldexp(1.0, -6)) {                     /* subnormal range: step 2^-9 */
    double m = rint(a * 512.0);                      /* exact scaling, RNE */
    if (m >= 8.0) code = (uint8_t)(1 << 3);          /* rounds up to min normal 2^-6 */
    else code = (uint8_t)m;
  } else {
    int ex;
    frexp(a, &ex);                                   /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                                  /* a in [2^e, 2^(e+1)) */
    double m = rint(ldexp(a, 3 - e));                /* in [8, 16], RNE */
    if (m >= 16.0) { m = 8.0; e += 1; }
    if (e > 8 || (e == 8 && m > 14.0)) code = 0x7E; /* above 448: saturate */
    else code = (uint8_t)(((e + 7) << 3) | ((int)m - 8));
  }
  return (uint8_t)(code | (s << 7));
}

void oc_e4m3_encode_array(const float* f, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oc_e4m3_encode(f[i]);
}

/* Block quantisation with fp32 scales (the FP8-dispatch variant: tokens in 1x128 blocks,  */
/* weights in 128x128 blocks; the pages name FP8 dispatch and FP8/FP4 training but no     */
/* block shape, and these are the reading taken). Per block: amax = max |v| (exact); if    */
/* amax == 0 the scale is 1 and every code is 0; else scale = amax / 448 and              */
/* q = e4m3(v * (448 / amax)), each                                                       */
/* division and the product one correctly rounded fp32 operation. The value the block      */
/* stands for is decode(q) * scale. scale is [rows/br][cols/bc] row-major.                 */
void oc_quant_blocks(const float* v, int64_t rows, int64_t cols, int br, int bc, uint8_t* q,
                     float* scale) {
  int64_t nbr = (rows + br - 1) / br, nbc = (cols + bc - 1) / bc;
#pragma omp parallel for schedule(static)
  for (int64_t bi = 0; bi < nbr * nbc; ++bi) {
    int64_t r0 = (bi / nbc) * br, c0 = (bi % nbc) * bc;
    int64_t r1 = r0 + br < rows ? r0 + br : rows, c1 = c0 + bc < cols ? c0 + bc : cols;
    float amax = 0.0f;
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t c = c0; c < c1; ++c) {
        float a = fabsf(v[r * cols + c]);
        if (a > amax) amax = a;
      }
    if (amax == 0.0f) {
      scale[bi] = 1.0f;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) q[r * cols + c] = 0;
    } else {
      volatile float sc = amax / 448.0f; /* volatile: keep each fp32 rounding */
      volatile float rs = 448.0f / amax;
      scale[bi] = sc;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) {
          volatile float p = v[r * cols + c] * rs;
          q[r * cols + c] = oc_e4m3_encode(p);
        }
    }
  }
}

/* decode(q) * scale in fp64 (the exact value of a quantised block). */
void oc_dequant_blocks(const uint8_t* q, const float* scale, int64_t rows, int64_t cols, int br,
                       int bc, double* out) {
  int64_t nbc = (cols + bc - 1) / bc;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = oc_e4m3_decode(q[r * cols + c]) * (double)scale[(r / br) * nbc + c / bc];
}

/* MX block quantisation (the MXFP8 format the Megatron-Core summary and the Hybrid-EP    */
/* article name for Blackwell; defined by the OCP Microscaling Formats (MX) specification */
/* v1.0, conversion of a block to MXFP8 E4M3). Every 32 consecutive values of a row share */
/* one power-of-two scale X = 2^s, stored as the UE8M0 code s + 127:                       */
/*   s = floor(log2(amax)) - 8   (8 = exponent of the largest e4m3 normal, 448 = 1.75*2^8) */
/* clamped to [-127, 127]; an all-zero block takes s = -127. Each element is              */
/* e4m3(v * 2^-s), a correctly rounded fp32 scaling by a power of two, encoded with RNE    */
/* and saturation to +-448, so the largest element of a block may saturate, as the         */
/* specification's conversion allows. cols is a multiple of 32; sc is [rows][cols/32].     */
void oc_mx_quant(const float* v, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sc) {
  int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t bi = 0; bi < rows * nb; ++bi) {
    const int64_t off = (bi / nb) * cols + (bi % nb) * 32;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      float a = fabsf(v[off + i]);
      if (a > amax) amax = a;
    }
    int s = -127;
    if (amax > 0.0f) {
      int ex;
      frexpf(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2(amax)) = ex - 1 */
      s = ex - 1 - 8;
      if (s < -127) s = -127;
      if (s > 127) s = 127;
    }
    sc[bi] = (uint8_t)(s + 127);
    for (int i = 0; i < 32; ++i) {
      volatile float p = ldexpf(v[off + i], -s);
      q[off + i] = oc_e4m3_encode(p);
    }
  }
}

/* decode(q) * 2^(code - 127) in fp64 (the exact value of an MX block). */
void oc_mx_dequant(const uint8_t* q, const uint8_t* sc, int64_t rows, int64_t cols, double* out) {
  int64_t nb = cols / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = ldexp(oc_e4m3_decode(q[r * cols + c]), (int)sc[r * nb + c / 32] - 127);
}

/* ------------------------------------------------------------------------------------ */
/* S4 + S5: one expert's SwiGLU MLP on a set of rows, fp64 (one expert's share of the     */
/* grouped GEMM of the Megatron-Core summary, section 2.4; SwiGLU from the workload       */
/* definition):                                                                           */
/*   g = a . Wg^T,  u = a . Wu^T,  h = g / (1 + e^-g) * u,  y = h . Wd^T.                 */
/* a is [n, H], Wg/Wu [F, H], Wd [H, F] (all fp64 values). quant_h 1: h is rounded to     */
/* fp32 and requantised in 1x128 blocks as the FP8-dispatch variant does before the down   */
/* projection; quant_h 2: the same in 1x32 MX blocks (MXFP8 variant). y then uses the      */
/* dequantised h.                                                                         */
/* ------------------------------------------------------------------------------------ */
void oc_expert_mlp(const double* a, int64_t n, int H, int F, const double* wg, const double* wu,
                   const double* wd, int quant_h, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    double* h = (double*)malloc(sizeof(double) * (size_t)F);
    const double* ar = a + r * H;
    for (int f = 0; f < F; ++f) {
      double g = 0.0, u = 0.0;
      const double* wgf = wg + (int64_t)f * H;
      const double* wuf = wu + (int64_t)f * H;
      for (int i = 0; i < H; ++i) { g += ar[i] * wgf[i]; u += ar[i] * wuf[i]; }
      h[f] = g / (1.0 + exp(-g)) * u;
    }
    if (quant_h == 1) {
      float* h32 = (float*)malloc(sizeof(float) * (size_t)F);
      uint8_t* q = (uint8_t*)malloc((size_t)F);
      float* sc = (float*)malloc(sizeof(float) * (size_t)((F + 127) / 128));
      for (int f = 0; f < F; ++f) h32[f] = (float)h[f];
      oc_quant_blocks(h32, 1, F, 1, 128, q, sc);
      for (int f = 0; f < F; ++f) h[f] = oc_e4m3_decode(q[f]) * (double)sc[f / 128];
      free(h32); free(q); free(sc);
    } else if (quant_h == 2) {
      float* h32 = (float*)malloc(sizeof(float) * (size_t)F);
      uint8_t* q = (uint8_t*)malloc((size_t)F);
      uint8_t* sc = (uint8_t*)malloc((size_t)(F / 32));
      for (int f = 0; f < F; ++f) h32[f] = (float)h[f];
      oc_mx_quant(h32, 1, F, q, sc);
      oc_mx_dequant(q, sc, 1, F, h);
      free(h32); free(q); free(sc);
    }
    for (int o = 0; o < H; ++o) {
      double s = 0.0;
      const double* wdo = wd + (int64_t)o * F;
      for (int f = 0; f < F; ++f) s += h[f] * wdo[f];
      y[r * H + o] = s;
    }
    free(h);
  }
}

/* ------------------------------------------------------------------------------------ */
/* S7: combine. y[t] = sum_j w[t,j] * yd[tok_row[t,j]] (+ ys[t], the shared expert's row) */
/* in fp64, w already holding the routed scale: the Hybrid-EP article's combine operator */
/* returns the expert outputs to token order and accumulates them in high precision;     */
/* dropless, every token gets all k rows (Megatron-Core summary, dropless MoE). ys may    */
/* be NULL.                                                                               */
/* ------------------------------------------------------------------------------------ */
void oc_combine(const double* yd, const int32_t* tok_row, const double* w, const double* ys,
                int T, int k, int H, double* y) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int o = 0; o < H; ++o) {
      double s = 0.0;
      for (int j = 0; j < k; ++j)
        s += w[(int64_t)t * k + j] * yd[(int64_t)tok_row[(int64_t)t * k + j] * H + o];
      if (ys) s += ys[(int64_t)t * H + o];
      y[(int64_t)t * H + o] = s;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Backward of the layer for a training step (the pages' grouped GEMM and permutation    */
/* serve the backward as well as the forward: Megatron-Core summary, section 2.4 grouped  */
/* GEMM and the memory-efficient permutation; section 2.2 recomputation of activations).  */
/* With the routing fixed (its map and weights are inputs here), y depends on x through   */
/* dispatch, the experts and combine; the functions below are the chain rule of those     */
/* steps, in fp64, in the reverse order.                                                 */
/* ------------------------------------------------------------------------------------ */

/* Backward of the auxiliary loss above, counts held fixed (they are integers): with      */
/* a_e = alpha * E * c_e / (T^2 * k) = dL/dp_hat[t,e] for every token, and p_hat the      */
/* normalised probabilities, adds to dl[t,:]                                              */
/*   softmax:  p_hat_e (a_e - sum_j a_j p_hat_j)                                          */
/*   sigmoid:  s_e (1 - s_e) (a_e - sum_j a_j p_hat_j) / sum_j s_j                         */
void oc_aux_loss_backward(const float* logits, const int32_t* counts, int T, int E, int k, int score_fn,
                          double alpha, double* dl) {
  if (T == 0) return;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    double* d = dl + (int64_t)t * E;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double sum = 0.0, c = 0.0;
    if (score_fn == 0) {
      double m = -INFINITY;
      for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
      for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - m); sum += p[e]; }
    } else {
      for (int e = 0; e < E; ++e) { p[e] = 1.0 / (1.0 + exp(-(double)l[e])); sum += p[e]; }
    }
    const double a0 = alpha * (double)E / ((double)T * (double)T * (double)k);
    for (int e = 0; e < E; ++e) c += a0 * (double)counts[e] * p[e] / sum;
    for (int e = 0; e < E; ++e) {
      const double de = a0 * (double)counts[e] - c;
      d[e] += score_fn == 0 ? p[e] / sum * de : p[e] * (1.0 - p[e]) * de / sum;
    }
    free(p);
  }
}

/* Router backward. The top-k choice is a piecewise-constant function of the logits and  */
/* is held fixed; the chosen weights are w = rho * f(l) with f the weight step of          */
/* route_one. With g[j] = rho * dw[t,j] (dw = dL/dw, the combine backward's result):        */
/*   softmax over all experts:  p = softmax(l);  dl[e] = [e chosen] g_e p_e - p_e sum_j g_j p_j */
/*   softmax over the chosen k: q = softmax(l over the chosen); dl[i_j] = q_j (g_j - sum g q) */
/*   sigmoid s, normalised:     w~ = s / S;  dl[i_j] = s_j (1 - s_j) (g_j - sum g w~) / S     */
/*   sigmoid, not normalised:   dl[i_j] = g_j s_j (1 - s_j)                                  */
/* and dl = 0 for experts not chosen, except in the first form. Experts chosen twice do  */
/* not occur (a token's k experts are distinct).                                          */
void oc_router_backward(const float* logits, int T, int E, int k, const int32_t* topk_idx, int score_fn,
                        int renorm, double routed_scale, const double* dw, double* dl) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    const int32_t* idx = topk_idx + (int64_t)t * k;
    double* d = dl + (int64_t)t * E;
    double* g = (double*)malloc(sizeof(double) * (size_t)k);
    double* v = (double*)malloc(sizeof(double) * (size_t)k);
    for (int e = 0; e < E; ++e) d[e] = 0.0;
    for (int j = 0; j < k; ++j) g[j] = routed_scale * dw[(int64_t)t * k + j];
    if (score_fn == 0) {
      double m = -INFINITY;
      for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
      if (renorm) {
        double den = 0.0, c = 0.0;
        for (int j = 0; j < k; ++j) { v[j] = exp((double)l[idx[j]] - m); den += v[j]; }
        for (int j = 0; j < k; ++j) { v[j] /= den; c += g[j] * v[j]; }
        for (int j = 0; j < k; ++j) d[idx[j]] = v[j] * (g[j] - c);
      } else {
        double den = 0.0, c = 0.0;
        for (int e = 0; e < E; ++e) den += exp((double)l[e] - m);
        for (int j = 0; j < k; ++j) { v[j] = exp((double)l[idx[j]] - m) / den; c += g[j] * v[j]; }
        for (int e = 0; e < E; ++e) d[e] = -exp((double)l[e] - m) / den * c;
        for (int j = 0; j < k; ++j) d[idx[j]] += g[j] * v[j];
      }
    } else {
      double S = 0.0, c = 0.0;
      for (int j = 0; j < k; ++j) { v[j] = 1.0 / (1.0 + exp(-(double)l[idx[j]])); S += v[j]; }
      if (renorm) {
        for (int j = 0; j < k; ++j) c += g[j] * v[j] / S;
        for (int j = 0; j < k; ++j) d[idx[j]] = v[j] * (1.0 - v[j]) * (g[j] - c) / S;
      } else {
        for (int j = 0; j < k; ++j) d[idx[j]] = g[j] * v[j] * (1.0 - v[j]);
      }
    }
    free(g);
    free(v);
  }
}

/* Combine backward. From y[t] = sum_j w[t,j] * yd[r_tj] (+ yd[R+t]):                    */
/*   dyd[r_tj] = w[t,j] * dy[t],  dyd[R+t] = dy[t]  (shared),                            */
/*   dw[t,j]  = sum_o dy[t,o] * yd[r_tj, o].                                              */
void oc_combine_backward(const double* dy, const double* yd, const int32_t* tok_row, const double* w,
                         int T, int k, int H, int shared, double* dyd, double* dw) {
  const int64_t R = (int64_t)T * k;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double* g = dy + (int64_t)t * H;
    for (int j = 0; j < k; ++j) {
      const int64_t r = tok_row[(int64_t)t * k + j];
      const double wj = w[(int64_t)t * k + j];
      double s = 0.0;
      for (int o = 0; o < H; ++o) {
        dyd[r * H + o] = wj * g[o];
        s += g[o] * yd[r * H + o];
      }
      dw[(int64_t)t * k + j] = s;
    }
    if (shared)
      for (int o = 0; o < H; ++o) dyd[(R + t) * H + o] = g[o];
  }
}

/* One expert's SwiGLU MLP backward on rows a [n,H] with output gradient dyd [n,H]. The  */
/* activations are recomputed from a (g = a Wg^T, u = a Wu^T, s = 1/(1+e^-g),            */
/* h = g s u), not stored:                                                              */
/*   dh  = dyd . Wd                 (dgrad of the down projection)                       */
/*   dg  = dh * u * s * (1 + g (1 - s)),  du = dh * g * s   (SwiGLU backward)            */
/*   dxd = dg . Wg + du . Wu        (dgrad of gate/up)                                   */
/*   dWd = dyd^T . h,  dWg = dg^T . a,  dWu = du^T . a   (wgrad, summed over the rows)   */
/* Outputs: dxd [n,H], dwg/dwu [F,H], dwd [H,F].                                         */
void oc_expert_mlp_backward(const double* a, int64_t n, int H, int F, const double* wg, const double* wu,
                            const double* wd, const double* dyd, double* dxd, double* dwg, double* dwu,
                            double* dwd) {
  double* h = (double*)malloc(sizeof(double) * (size_t)(n * F > 0 ? n * F : 1));
  double* dg = (double*)malloc(sizeof(double) * (size_t)(n * F > 0 ? n * F : 1));
  double* du = (double*)malloc(sizeof(double) * (size_t)(n * F > 0 ? n * F : 1));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    const double* ar = a + r * H;
    const double* gy = dyd + r * H;
    for (int f = 0; f < F; ++f) {
      double g = 0.0, u = 0.0, dh = 0.0;
      for (int i = 0; i < H; ++i) {
        g += ar[i] * wg[(int64_t)f * H + i];
        u += ar[i] * wu[(int64_t)f * H + i];
      }
      for (int o = 0; o < H; ++o) dh += gy[o] * wd[(int64_t)o * F + f];
      const double s = 1.0 / (1.0 + exp(-g));
      h[r * F + f] = g * s * u;
      dg[r * F + f] = dh * u * s * (1.0 + g * (1.0 - s));
      du[r * F + f] = dh * g * s;
    }
    for (int i = 0; i < H; ++i) {
      double x = 0.0;
      for (int f = 0; f < F; ++f) x += dg[r * F + f] * wg[(int64_t)f * H + i] + du[r * F + f] * wu[(int64_t)f * H + i];
      dxd[r * H + i] = x;
    }
  }
#pragma omp parallel for schedule(static)
  for (int o = 0; o < H; ++o)
    for (int f = 0; f < F; ++f) {
      double x = 0.0;
      for (int64_t r = 0; r < n; ++r) x += dyd[r * H + o] * h[r * F + f];
      dwd[(int64_t)o * F + f] = x;
    }
#pragma omp parallel for schedule(static)
  for (int f = 0; f < F; ++f)
    for (int i = 0; i < H; ++i) {
      double xg = 0.0, xu = 0.0;
      for (int64_t r = 0; r < n; ++r) {
        xg += dg[r * F + f] * a[r * H + i];
        xu += du[r * F + f] * a[r * H + i];
      }
      dwg[(int64_t)f * H + i] = xg;
      dwu[(int64_t)f * H + i] = xu;
    }
  free(h); free(dg); free(du);
}

/* Dispatch backward: dx[t] = sum_j dxd[r_tj] (+ dxd[R+t]): every copy of a token sends   */
/* its gradient back to the token.                                                       */
void oc_dispatch_backward(const double* dxd, const int32_t* tok_row, int T, int k, int H, int shared,
                          double* dx) {
  const int64_t R = (int64_t)T * k;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int i = 0; i < H; ++i) {
      double s = 0.0;
      for (int j = 0; j < k; ++j) s += dxd[(int64_t)tok_row[(int64_t)t * k + j] * H + i];
      if (shared) s += dxd[(R + t) * H + i];
      dx[(int64_t)t * H + i] = s;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Second, independent oracle: the dense per-token loop. For each token, re-derive the    */
/* top-k from its fp32 logits and run the chosen experts directly, with no counts, no     */
/* permutation and no dispatch buffer. Weights in fp64 (Wg/Wu [E,F,H], Wd [E,H,F]).        */
/* Shared expert optional (wsg/wsu [Fs,H], wsd [H,Fs], may be NULL).                       */
/* ------------------------------------------------------------------------------------ */
int oc_dense_forward(const double* x, const float* logits, int T, int H, int E, int k, int F,
                     int score_fn, int renorm, int n_groups, int topk_groups, int group_score,
                     double rho, const double* wg, const double* wu, const double* wd,
                     int Fs, const double* wsg, const double* wsu, const double* wsd,
                     double* y) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int t = 0; t < T; ++t) {
    int32_t idx[1024];
    double w[1024];
    if (route_one(logits + (int64_t)t * E, E, k, score_fn, renorm, n_groups, topk_groups,
                  group_score, rho, idx, w, NULL)) { bad = 1; continue; }
    const double* xt = x + (int64_t)t * H;
    double* yt = y + (int64_t)t * H;
    for (int o = 0; o < H; ++o) yt[o] = 0.0;
    int nexp = k + (wsg ? 1 : 0);
    for (int j = 0; j < nexp; ++j) {
      int shared = (j == k);
      int FF = shared ? Fs : F;
      const double* G = shared ? wsg : wg + (int64_t)idx[j] * F * H;
      const double* U = shared ? wsu : wu + (int64_t)idx[j] * F * H;
      const double* D = shared ? wsd : wd + (int64_t)idx[j] * H * F;
      double c = shared ? 1.0 : w[j];
      double* h = (double*)malloc(sizeof(double) * (size_t)FF);
      for (int f = 0; f < FF; ++f) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < H; ++i) { g += xt[i] * G[(int64_t)f * H + i]; u += xt[i] * U[(int64_t)f * H + i]; }
        h[f] = g / (1.0 + exp(-g)) * u;
      }
      for (int o = 0; o < H; ++o) {
        double s = 0.0;
        for (int f = 0; f < FF; ++f) s += h[f] * D[(int64_t)o * FF + f];
        yt[o] += c * s;
      }
      free(h);
    }
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------ */
/* Auxiliary load-balancing loss (Megatron-Core skill card, Fluxo 2: the "aux_loss" load */
/* balancing type with --moe-aux-loss-coeff 0.01; the pages give no formula). Reading:    */
/* the switch-style loss  L = alpha * E / (T*k) * sum_e c_e * Pbar_e,  c_e the routed      */
/* count of expert e and Pbar_e the mean over tokens of the token's probability for e:    */
/* the softmax over all experts (score_fn 0) or the sigmoid scores divided by their sum    */
/* over all experts (score_fn 1). fp64.                                                   */
/* ------------------------------------------------------------------------------------ */
double oc_aux_loss(const float* logits, const int32_t* counts, int T, int E, int k, int score_fn,
                   double alpha, double* pbar_out) {
  double* pbar = (double*)calloc((size_t)E, sizeof(double));
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (int64_t)t * E;
    double sum = 0.0;
    if (score_fn == 0) {
      double m = -INFINITY;
      for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
      for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - m); sum += p[e]; }
    } else {
      for (int e = 0; e < E; ++e) { p[e] = 1.0 / (1.0 + exp(-(double)l[e])); sum += p[e]; }
    }
    for (int e = 0; e < E; ++e) pbar[e] += p[e] / sum;
  }
  double loss = 0.0;
  for (int e = 0; e < E; ++e) {
    pbar[e] /= (double)T;
    if (pbar_out) pbar_out[e] = pbar[e];
    loss += (double)counts[e] * pbar[e];
  }
  loss *= alpha * (double)E / ((double)T * (double)k);
  free(p);
  free(pbar);
  return loss;
}
