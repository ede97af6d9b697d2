/*
 * moe.h — C ABI of the GB300 (sm_103a) single-GPU Mixture-of-Experts layer forward.
 *
 * The layer, as the method states it: a router scores every token against the experts
 * and activates k of them ("Scalable Training of Mixture-of-Experts Models with Megatron
 * Core" summary, "O essencial"); dispatch directs each token to its experts and combine
 * sends the results back, accumulating in high precision (Hybrid-EP article, dispatch and
 * combine operators); the experts' GEMMs run together as one grouped GEMM (Megatron-Core
 * summary, section 2.4 "Grouped GEMM"); routing is dropless, and kernels read the dynamic
 * per-expert shapes from device memory so that no host synchronisation is needed
 * (section 2.4, "Kernels Iniciados pelo Dispositivo"; Hybrid-EP article, pre-sized
 * buffers). On one GPU, dispatch and combine are on-device permutations.
 *
 *   moe_router_logits   S0  logits[t,e] = sum_h x[t,h] * Wr[e,h] (+ bias[e])
 *   moe_route           S1  top-k (optionally group-limited) + weights, then S2
 *   moe_route_from_map  S2  counts, offsets and the permutation from a given map (replay)
 *   moe_dispatch        S3  xd[r] = x[row_token[r]] (FP8: quantised once per token)
 *   moe_dispatch_mx     S3  the same for the MXFP8 variant (1x32 blocks, UE8M0 scales)
 *   moe_grouped_mlp     S4-S6  per expert: h = silu(xd Wg^T) * (xd Wu^T); yd = h Wd^T
 *   moe_combine         S7  y[t] = sum_j w[t,j] * yd[tok_row[t,j]] (+ shared row)
 *   moe_forward         S0-S7 in one stream-ordered call
 *   moe_forward_host    the same with the tokens and the output in host memory
 *   moe_backward        the training step's backward of S0-S7 (bf16 layers): combine,
 *                       the experts' grouped dgrad/wgrad with recomputed SwiGLU, dispatch,
 *                       and (optionally) the router and the auxiliary loss
 *   moe_forward_train   moe_forward that keeps the gate/up pre-activations, and
 *   moe_backward_kept   the backward that reads them instead of rerunning that GEMM
 *   moe_router_backward the router's backward: dlogits, dW_router, d bias
 *
 * Conventions shared by every call:
 *  - Every data pointer is DEVICE memory owned by the caller; the library allocates
 *    nothing and frees nothing. Pointers must be 16-byte aligned.
 *  - Every matrix is row-major and dense (leading dimension = its column count).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL means the legacy default
 *    stream) and never synchronise the host, except moe_read_status.
 *  - The return code covers host-side validation and launch errors only. Faults found on
 *    the device (an expert id out of range in a replayed map, a non-finite router score,
 *    a bounded wait that expired) are written to a status word in the workspace; read it
 *    with moe_read_status.
 *  - Re-entrant as long as two calls in flight at once do not share a workspace.
 *
 * Shapes: T tokens, H hidden, E routed experts, k experts per token, F expert FFN width.
 * R = T*k routed rows; with a shared expert the dispatch/expert buffers hold R + T rows,
 * the shared expert's row for token t being row R + t.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, inconsistent sizes */
  MOE_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. H % 64 != 0 on bf16) */
  MOE_ERR_CUDA = 3,             /* a CUDA launch or driver call failed */
  MOE_ERR_DEVICE_BAD_INPUT = 4, /* device status: id out of range or non-finite score */
  MOE_ERR_TIMEOUT = 5           /* device status: a bounded wait in a kernel expired */
} moe_status_t;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
/* MOE_DTYPE_E4M3: e4m3 with fp32 scales per 1x128 (activations) / 128x128 (weights) block.
 * MOE_DTYPE_MXE4M3: MXFP8 (OCP Microscaling v1.0): e4m3 with one power-of-two UE8M0 scale
 * per 1x32 block of every row, stored in scale atoms (below). */
enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1, MOE_DTYPE_E4M3 = 2, MOE_DTYPE_MXE4M3 = 3 };
enum { MOE_GROUP_SCORE_TOP2_SUM = 0, MOE_GROUP_SCORE_MAX = 1 };

/* Layer configuration: plain values, no pointers. */
typedef struct {
  int32_t T, H, E, k, F;
  int32_t n_shared;    /* 0 or 1 shared expert, applied to every token with weight 1 */
  int32_t F_shared;    /* its FFN width; must equal F when n_shared = 1 */
  int32_t score_fn;    /* MOE_SCORE_SOFTMAX or MOE_SCORE_SIGMOID */
  int32_t renorm;      /* 1: weights normalised over the k selected experts */
  int32_t n_groups;    /* G: experts split into G contiguous groups (1 = no grouping) */
  int32_t topk_groups; /* g: groups kept before the top-k (g = G: no limit); sigmoid only */
  int32_t group_score; /* MOE_GROUP_SCORE_*: sum of the two largest scores, or the max */
  float routed_scale;  /* every routed weight is multiplied by this (1.0) */
  int32_t act_dtype;   /* MOE_DTYPE_F32 or MOE_DTYPE_BF16: x, router and (unless E4M3) expert weights, y */
  int32_t xfer_dtype;  /* = act_dtype, or MOE_DTYPE_E4M3 / MOE_DTYPE_MXE4M3 (bf16 act only): dispatched rows and expert GEMMs in e4m3 */
} moe_config_t;

/* Layer weights (device pointers). act = act_dtype; q = e4m3 when xfer_dtype is E4M3 or
 * MXE4M3, else act. E4M3 weights carry fp32 scales per 128x128 block (value = code *
 * scale, [rows/128, cols/128] row-major); MXE4M3 weights carry the UE8M0 scale atoms of
 * their rows (moe_quantize_mx: tile a = rows [128a, 128a + 128)). The s_* / ss_* fields are
 * NULL for unquantised layers. */
typedef struct {
  const void* w_router;     /* [E, H] act */
  const float* router_bias; /* [E] fp32 added to every logit, or NULL */
  const void* w_gate;       /* [E, F, H] q */
  const void* w_up;         /* [E, F, H] q */
  const void* w_down;       /* [E, H, F] q */
  const void* s_gate;       /* E4M3: fp32 [E, F/128, H/128]; MXE4M3: atoms of [E*F, H] */
  const void* s_up;         /* E4M3: fp32 [E, F/128, H/128]; MXE4M3: atoms of [E*F, H] */
  const void* s_down;       /* E4M3: fp32 [E, H/128, F/128]; MXE4M3: atoms of [E*H, F] */
  const void* ws_gate;      /* shared expert [F, H] q, or NULL when n_shared = 0 */
  const void* ws_up;        /* [F, H] q */
  const void* ws_down;      /* [H, F] q */
  const void* ss_gate;      /* E4M3: fp32 [F/128, H/128]; MXE4M3: atoms of [F, H] */
  const void* ss_up;        /* E4M3: fp32 [F/128, H/128]; MXE4M3: atoms of [F, H] */
  const void* ss_down;      /* E4M3: fp32 [H/128, F/128]; MXE4M3: atoms of [H, F] */
} moe_weights_t;

/* Weight gradients written by the backward (device fp32, caller-owned; overwritten, not
 * accumulated). The router fields are optional: with dw_router = NULL, moe_backward leaves
 * the router out and its dx holds the gradient through the experts only. */
typedef struct {
  float* dw_gate;       /* [E, F, H] */
  float* dw_up;         /* [E, F, H] */
  float* dw_down;       /* [E, H, F] */
  float* dws_gate;      /* shared expert [F, H], or NULL when n_shared = 0 */
  float* dws_up;        /* [F, H] */
  float* dws_down;      /* [H, F] */
  float* dw_router;     /* [E, H], or NULL: no router backward */
  float* d_router_bias; /* [E], or NULL: not written (the column sums of dlogits) */
  float* dlogits;       /* [T, E], or NULL: kept in the backward workspace */
  float aux_loss_coeff; /* alpha of moe_aux_loss, whose gradient joins dlogits; 0: none */
} moe_weight_grads_t;

/* MX scale atoms. The UE8M0 codes (code = s + 127 for the block scale 2^s) of an e4m3
 * matrix with K columns (K a multiple of 128) are stored in 512-byte atoms, each covering
 * 128 rows ("tile" a) and one 128-column K stage ks (four 1x32 blocks kb = 0..3): atom
 * (a, ks) begins at byte (a * (K/128) + ks) * 512, and the code of the tile's row i and
 * block kb is at byte (i % 32) * 16 + (i / 32) * 4 + kb of the atom. This is the order in
 * which the block-scaled tensor-core MMA reads scale factors, so one copy per atom feeds it.
 *  - Weights: tile a holds rows [128a, 128a + 128).
 *  - Grouped activations (dispatched rows, h): the rows of expert e (e = E: the shared
 *    expert, whose offset is offsets[E] = T*k) start a fresh tile at
 *    base(e) = ceil((offsets[e] + 127 * e) / 128), and row r of expert e is row
 *    (r - offsets[e]) % 128 of tile base(e) + (r - offsets[e]) / 128. The buffer size
 *    comes from moe_mx_scale_bytes. Tile rows past an expert's last row are never written
 *    and never read into a result. */

/* Bytes of device workspace needed by every call below except moe_forward (the status
 * word, the routing scan's per-block counts and the auxiliary loss's per-block sums). Zero
 * it once with moe_workspace_init. */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Bytes of device workspace for moe_forward: the part above followed by every
 * intermediate of the layer (logits, routing map, permutation, dispatched rows, h, yd). */
moe_status_t moe_forward_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Clears the head of a workspace (its status word and the routing kernel's grid barrier;
 * stream-ordered). Call once after allocating, and again after a failed call. */
moe_status_t moe_workspace_init(void* ws, moe_stream_t stream);

/* S0 — router logits (Megatron-Core summary, "O essencial": the router scores each token
 * against every expert). x [T,H] act, w_router [E,H] act, router_bias [E] fp32 or NULL ->
 * logits [T,E] fp32, accumulated in fp32. */
moe_status_t moe_router_logits(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, float* logits, void* ws,
                               moe_stream_t stream);

/* S1 + S2 — routing. From fp32 scores `logits` [T,E]: per token the k experts with the
 * largest logit (ties to the lower expert index), after keeping only the topk_groups best
 * groups when n_groups > 1 (group score from sigmoid scores computed with a fixed,
 * machine-independent fp32 exp). Outputs:
 *   topk_idx [T,k] int32, in descending key order;
 *   topk_w   [T,k] fp32: softmax (over all experts, or the k selected when renorm) or
 *            sigmoid (divided by the selected sum when renorm), times routed_scale;
 *   counts [E], offsets [E+1] int32 (offsets[E] = T*k);
 *   row_token [T*k]: the token in each dispatched row, rows of expert e being
 *            [offsets[e], offsets[e+1]) in ascending token id;
 *   tok_row [T,k]: the row holding token t's j-th choice.
 * Bit-exact and deterministic (no atomics whose order shows in the result).
 * A non-finite logit sets MOE_ERR_DEVICE_BAD_INPUT in the status word.
 * One cooperative launch (every block resident at once) routes contiguous token chunks,
 * publishes their per-expert counts in the workspace and, after a grid barrier kept in the
 * workspace head (and, with more than 8192 per-block counts, a scan of each expert's counts
 * and a second barrier), writes the map. A barrier's wait is bounded: if it gives up,
 * MOE_ERR_TIMEOUT is set and the map is left empty (counts and offsets zero, tok_row 0). */
moe_status_t moe_route(const moe_config_t* cfg, const float* logits, int32_t* topk_idx,
                       float* topk_w, int32_t* counts, int32_t* offsets, int32_t* row_token,
                       int32_t* tok_row, void* ws, moe_stream_t stream);

/* The number of kernel launches moe_route makes for this configuration (0 when T = 0): 1
 * for the cooperative launch, else the top-k launch and the scan (one launch up to 512
 * tokens, else three). The cooperative launch is taken where a block's token chunk times
 * ceil(E / 32) is at most 1024, which depends on the device's occupancy for the kernel
 * (queried here on first use of a shape). Launches nothing. */
moe_status_t moe_route_launch_count(const moe_config_t* cfg, int32_t* launches);

/* S2 only, from a given routing map (router replay, Megatron-Core summary section 2.5).
 * An id outside [0,E) sets MOE_ERR_DEVICE_BAD_INPUT; that entry is then counted for
 * expert 0 so that every output stays in bounds. */
moe_status_t moe_route_from_map(const moe_config_t* cfg, const int32_t* topk_idx,
                                int32_t* counts, int32_t* offsets, int32_t* row_token,
                                int32_t* tok_row, void* ws, moe_stream_t stream);

/* Auxiliary load-balancing loss of the routing (Megatron-Core skill card, Fluxo 2:
 * load-balancing type "aux_loss" with --moe-aux-loss-coeff, 0.01 there; the pages give no
 * formula, so the switch-style form is taken):
 *   loss = alpha * E / (T*k) * sum_e counts[e] * Pbar_e,
 * Pbar_e = the mean over tokens of expert e's probability: the softmax of the token's logits
 * over all experts, or its sigmoid scores divided by their sum (score_fn). A non-finite
 * logit counts as -FLT_MAX, as in routing. Each token's probability is rounded to a multiple
 * of 2^-32 and the sums over tokens, and sum_e counts[e] * (that sum), are exact integers
 * (64 and 128 bits), so the value does not depend on how the work is split: moe_forward_train
 * gives the same bits from inside its routing. logits [T,E] fp32, counts [E] from moe_route;
 * *loss is one device float. Uses the workspace's scratch (stream-ordered after moe_route on
 * the same workspace is fine). Deterministic. */
moe_status_t moe_aux_loss(const moe_config_t* cfg, const float* logits, const int32_t* counts,
                          float alpha, float* loss, void* ws, moe_stream_t stream);

/* S3 — dispatch (Hybrid-EP article, dispatch operator): xd[tok_row[t,j]] = x[t], reading
 * each token once. act xfer: xd [R(+T), H] act, bit copy; xd_scale unused (NULL).
 * E4M3 xfer: each token is quantised once in 1x128 blocks (scale = amax/448, codes =
 * e4m3_rn_satfinite(v * (448/amax)); an all-zero block has scale 1) and written to its k
 * rows (and row R+t with a shared expert); xd [R(+T), H] e4m3, xd_scale [H/128, R(+T)]
 * fp32 (block-major: scale of row r, block b at b*(R(+T)) + r). */
moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* tok_row,
                          void* xd, float* xd_scale, moe_stream_t stream);

/* S3 for the MXFP8 variant (xfer_dtype = MOE_DTYPE_MXE4M3; moe_dispatch returns
 * MOE_ERR_UNSUPPORTED for it). Each token is quantised once in 1x32 blocks (OCP MX v1.0:
 * s = floor(log2(amax)) - 8 clamped to [-127, 127], s = -127 for an all-zero block; codes
 * e4m3_rn_satfinite(v * 2^-s)) and written to its k rows xd[tok_row[t,j]] and, with a
 * shared expert, to row R + t; the UE8M0 codes go to the rows' places in the scale atoms
 * xd_sf (layout above: needs the expert of each row, hence topk_idx [T,k] and offsets
 * [E+1] from moe_route). xd [R(+T), H] e4m3; xd_sf moe_mx_scale_bytes(cfg, H, ...) bytes.
 * H % 128 == 0. A routed row whose expert id is outside [0, E) gets no scales. */
moe_status_t moe_dispatch_mx(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                             const int32_t* tok_row, const int32_t* offsets, void* xd, void* xd_sf,
                             moe_stream_t stream);

/* Bytes of an MX scale-atom buffer for the grouped activations of `cfg` with K columns
 * (K = H for moe_dispatch_mx's xd_sf, K = F for moe_grouped_mlp's h_scale). K % 128 == 0. */
moe_status_t moe_mx_scale_bytes(const moe_config_t* cfg, int32_t K, size_t* bytes);

/* S4 + S5 + S6 — the experts as one grouped GEMM (Megatron-Core summary section 2.4).
 * For expert e, rows r in [offsets[e], offsets[e+1]) of xd:
 *     h[r]  = silu(xd[r] . Wg[e]^T) * (xd[r] . Wu[e]^T),  silu(z) = z / (1 + e^-z)
 *     yd[r] = h[r] . Wd[e]^T
 * and, with a shared expert, the same for rows R + t with A = x[t] (act xfer) or the
 * dispatched row R + t (E4M3 / MXE4M3 xfer) and weights ws_*. The per-expert row counts
 * are read on the device; empty experts cost nothing. h [R(+T), F] act, or e4m3 (E4M3 /
 * MXE4M3 xfer) requantised from fp32 before the down projection: in 1x128 blocks with
 * h_scale fp32 [F/128, R(+T)] (E4M3), or in 1x32 MX blocks with h_scale the scale atoms
 * of h (MXE4M3, moe_mx_scale_bytes(cfg, F, ...) bytes); yd [R(+T), H] act. xd_scale: the
 * dispatched rows' scales (fp32 [H/128, R(+T)] for E4M3, atoms for MXE4M3), NULL otherwise.
 * MXE4M3 runs the block-scaled tensor-core MMA (the hardware applies the scales) and needs
 * H % 256 == 0, F % 128 == 0. `x` may be NULL unless act xfer with a shared expert. */
moe_status_t moe_grouped_mlp(const moe_config_t* cfg, const void* xd, const void* xd_scale,
                             const void* x, const int32_t* offsets, const moe_weights_t* w,
                             void* h, void* h_scale, void* yd, void* ws, moe_stream_t stream);

/* S3 + S4 + S5 fused — the grouped expert MLP with the dispatch folded into GEMM1's operand
 * loads: the memory-efficient permutation of the Megatron-Core summary (section 2.2: the
 * computation is reorganised so that no redundant intermediate tensor is materialised).
 * Routed A rows are gathered from x by token (row r reads x[row_token[r]]), so no
 * dispatched copy xd exists; the shared expert reads x directly. 256-row CTA-pair tiles
 * gather four rows per TMA instruction; 128-row single-CTA tiles copy their rows with
 * cp.async, eight lanes per row. Same outputs as moe_dispatch + moe_grouped_mlp
 * (bit-identical). bf16 layers on the tensor-core path only (else MOE_ERR_UNSUPPORTED).
 * x [T,H], row_token [T*k], offsets [E+1], h [R(+T), F], yd [R(+T), H]. moe_forward keeps
 * the separate dispatch: the gathers are slower on GB300 than the dispatch pass they
 * replace.
 * The other half of the fused permutation is optional: with tok_row [T,k] and topk_w [T,k]
 * (both given, or both NULL; else MOE_ERR_INVALID_ARG) the down projection's epilogue
 * scales each routed row by its routing weight before rounding,
 *     yd[r] = bf16(topk_w[t,j] * (h[r] . Wd[e]^T)),  t = row_token[r], tok_row[t,j] = r,
 * (shared-expert rows unweighted), and moe_combine with topk_w = NULL finishes the layer. */
moe_status_t moe_grouped_mlp_gather(const moe_config_t* cfg, const void* x, const int32_t* row_token,
                                    const int32_t* offsets, const int32_t* tok_row, const float* topk_w,
                                    const moe_weights_t* w, void* h, void* yd, void* ws,
                                    moe_stream_t stream);

/* S7 — combine (Hybrid-EP article, combine operator with high-precision accumulation):
 * y[t] = sum_{j<k} topk_w[t,j] * yd[tok_row[t,j]]  (+ yd[R + t] with a shared expert),
 * accumulated in fp32 in that fixed order, written once in act dtype. topk_w = NULL means
 * unit weights: the plain sum, for rows already weighted by moe_grouped_mlp_gather. */
moe_status_t moe_combine(const moe_config_t* cfg, const void* yd, const int32_t* tok_row,
                         const float* topk_w, void* y, moe_stream_t stream);

/* S0..S7 — the whole layer forward, stream-ordered with no host synchronisation, so the
 * call can be captured in a CUDA graph. ws: moe_forward_workspace_size bytes. The optional
 * outputs (NULL to skip) receive copies of the routing map and counts. */
moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const moe_weights_t* w,
                         void* y, void* ws, int32_t* topk_idx_out, float* topk_w_out,
                         int32_t* counts_out, moe_stream_t stream);

/* S0..S7 with the tokens and the output in host memory: x_host [T,H] is copied to x_dev,
 * moe_forward runs on it into y_dev, and y_dev is copied back to y_host, all three steps
 * stream-ordered on `stream`, so a caller can run the copies of one call under the kernels
 * of another issued on a second stream (with its own ws, x_dev and y_dev). x_host and y_host
 * are host memory; page-locked memory keeps the copies asynchronous (with pageable memory
 * the results are the same but the copies block the calling thread). x_dev, y_dev: device
 * buffers of T*H act-dtype elements, 16-byte aligned; ws as for moe_forward. The library
 * allocates nothing. Bit-identical to the copies around moe_forward. */
moe_status_t moe_forward_host(const moe_config_t* cfg, const void* x_host, const moe_weights_t* w,
                              void* y_host, void* x_dev, void* y_dev, void* ws, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Backward (a training step; bf16 layers on the tensor-core path, H % 256 == 0 and
 * F % 256 == 0, else MOE_ERR_UNSUPPORTED). The routing (map, weights, permutation) is that
 * of the forward and is held fixed: these calls return the gradient of the layer output with
 * respect to x through the experts, to the routing weights and to the expert weights, and
 * (moe_router_backward, moe_dispatch_router_backward) through the router to its logits, its
 * weight and bias and x. The experts' grouped
 * GEMMs serve the backward as in the forward (Megatron-Core summary, section 2.4), and the
 * SwiGLU activation is recomputed from the dispatched rows instead of being kept from the
 * forward (section 2.2, recomputation).
 * --------------------------------------------------------------------------------------- */

/* Bytes of workspace for moe_grouped_mlp_backward and moe_backward: the status head, then
 * dyd and dxd [R(+T), H], g/u and their gradients [R(+T), 2F], and h [R(+T), F], all bf16.
 * Zero it once with moe_workspace_init (its status word). */
moe_status_t moe_backward_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Combine backward: from the output gradient dy [T,H] and the forward's yd [R(+T), H],
 *   dyd[tok_row[t,j]] = topk_w[t,j] * dy[t],  dyd[R + t] = dy[t] (shared expert),
 *   dtopk_w[t,j] = sum_o dy[t,o] * yd[tok_row[t,j], o]   (fp32, the routing-weight gradient).
 * dyd [R(+T), H] bf16. */
moe_status_t moe_combine_backward(const moe_config_t* cfg, const void* dy, const void* yd,
                                  const int32_t* tok_row, const float* topk_w, void* dyd,
                                  float* dtopk_w, moe_stream_t stream);

/* The experts' backward as grouped GEMMs on the tensor cores, per expert e over its rows
 * (and the shared expert over rows R + t with input x[t]): g, u = xd Wg^T, xd Wu^T are
 * recomputed; dh = dyd Wd; dg = dh u s (1 + g (1 - s)), du = dh g s with s = sigmoid(g);
 * dxd = dg Wg + du Wu; dWd[e] = dyd^T h with h = g s u; dWg[e] = dg^T xd; dWu[e] = du^T xd
 * (sums over the expert's rows; an expert without rows gets zero gradients). xd [R, H] are
 * the forward's dispatched rows, x [T, H] the tokens (read for the shared expert), dyd from
 * moe_combine_backward; dxd [R(+T), H] bf16; grads fp32. ws: moe_backward_workspace_size. */
moe_status_t moe_grouped_mlp_backward(const moe_config_t* cfg, const void* xd, const void* x,
                                      const int32_t* offsets, const moe_weights_t* w, const void* dyd,
                                      void* dxd, const moe_weight_grads_t* grads, void* ws,
                                      moe_stream_t stream);

/* Dispatch backward: dx[t] = sum_j dxd[tok_row[t,j]] (+ dxd[R + t]), fp32 in that order,
 * written once in bf16 (the combine kernel with unit weights). */
moe_status_t moe_dispatch_backward(const moe_config_t* cfg, const void* dxd, const int32_t* tok_row,
                                   void* dx, moe_stream_t stream);

/* The three calls above in one stream-ordered call after moe_forward: the routing, the
 * dispatched rows and yd are read from that call's workspace fwd_ws (so it must not have
 * been reused in between), x and w are the forward's inputs, dy [T,H] bf16. Writes
 * dx [T,H] bf16, dtopk_w [T,k] fp32 and the weight gradients. With grads->dw_router set it
 * also runs the router's backward below on the forward's logits, map and counts (adding the
 * auxiliary loss's gradient when grads->aux_loss_coeff != 0) and forms dx with
 * moe_dispatch_router_backward, so that dx holds both shares. bwd_ws:
 * moe_backward_workspace_size bytes. */
moe_status_t moe_backward(const moe_config_t* cfg, const void* x, const moe_weights_t* w,
                          const void* dy, const void* fwd_ws, void* dx, float* dtopk_w,
                          const moe_weight_grads_t* grads, void* bwd_ws, moe_stream_t stream);

/* The forward of a training step: moe_forward, with GEMM1 also storing the gate/up
 * pre-activations g = xd Wg^T and u = xd Wu^T (bf16) into gu [R(+T), 2F], row r holding
 * F/128 blocks of 256 columns (128 of g, then 128 of u). With them kept, the backward
 * recomputes only the activation silu(g) u and its derivative, the cheap part (Megatron-Core
 * summary, section 2.2, granular recomputation: activation functions are recomputed rather
 * than stored), instead of rerunning the gate/up GEMM. gu is caller-owned: R(+T) * 2F * 2
 * bytes, 16-byte aligned. bf16 layers the backward takes (else MOE_ERR_UNSUPPORTED); y and
 * the workspace are bit-identical to moe_forward's. aux_loss: NULL, or one device float
 * that receives moe_aux_loss's loss (coefficient aux_alpha; a NaN coefficient is
 * MOE_ERR_INVALID_ARG) on this call's logits and counts (0 when T = 0); pass the same
 * coefficient as grads->aux_loss_coeff to moe_backward_kept for its gradient. Where routing
 * is one launch (moe_route_launch_count reports 1) that launch also forms the loss, reading
 * the logits once; otherwise two more launches after the routing do. */
moe_status_t moe_forward_train(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y, void* ws,
                               void* gu, float aux_alpha, float* aux_loss, moe_stream_t stream);

/* moe_backward after moe_forward_train: reads the kept gu instead of recomputing it. The
 * kept values are the ones the recomputation would produce, so every output is
 * bit-identical to moe_backward's. */
moe_status_t moe_backward_kept(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                               const void* fwd_ws, const void* gu, void* dx, float* dtopk_w,
                               const moe_weight_grads_t* grads, void* bwd_ws, moe_stream_t stream);

/* Router backward (the router scores every token against the experts, Megatron-Core
 * summary, "O essencial"; the weights are the softmax or sigmoid of the chosen scores).
 * The chosen experts are held fixed, so with g = routed_scale * dtopk_w[t, :]:
 *   softmax, not renormalised (p = softmax of all E logits):
 *       dlogits[t, e] = [e chosen as j] g_j p_e - p_e * sum_j g_j p_{i_j}
 *   softmax renormalised over the chosen (q_j = their softmax):
 *       dlogits[t, i_j] = q_j (g_j - sum_i g_i q_i)
 *   sigmoid s, renormalised (S = sum of the chosen s):
 *       dlogits[t, i_j] = s_j (1 - s_j) (g_j - sum_i g_i s_i / S) / S
 *   sigmoid, not renormalised:  dlogits[t, i_j] = g_j s_j (1 - s_j)
 * (zero for experts not chosen, except in the first form). With counts != NULL the
 * gradient of moe_aux_loss's loss (coefficient aux_alpha, counts held fixed) is added:
 *   a_e = aux_alpha * E * counts[e] / (T^2 k),  p_hat the loss's normalised probabilities,
 *   softmax: p_hat_e (a_e - sum a p_hat);  sigmoid: s_e (1 - s_e) (a_e - sum a p_hat) / sum s.
 * Then, for the linear router logits = x W_router^T (+ bias):
 *   dw_router[e, h] = sum_t dlogits[t, e] x[t, h],  d_router_bias[e] = sum_t dlogits[t, e],
 * summed in fp32 over token slices whose partial sums are added in a fixed order.
 * logits [T,E] fp32 (moe_router_logits), topk_idx [T,k] (moe_route; an id out of range sets
 * MOE_ERR_DEVICE_BAD_INPUT in the status word and leaves that token's row unwritten),
 * dtopk_w [T,k] fp32 (moe_combine_backward), x [T,H] act dtype, H % 8 == 0 (else
 * MOE_ERR_UNSUPPORTED). Outputs fp32: dlogits [T,E]; dw_router [E,H] or NULL (then x may be
 * NULL and no weight gradient is formed); d_router_bias [E] or NULL.
 * ws: moe_router_backward_workspace_size bytes (status head, partial sums, and on the
 * tensor-core path below dlogits in bf16 and the router's share of dx), initialised with
 * moe_workspace_init. */
moe_status_t moe_router_backward_workspace_size(const moe_config_t* cfg, size_t* bytes);
moe_status_t moe_router_backward(const moe_config_t* cfg, const float* logits, const int32_t* topk_idx,
                                 const float* dtopk_w, const int32_t* counts, float aux_alpha, const void* x,
                                 float* dlogits, float* dw_router, float* d_router_bias, void* ws,
                                 moe_stream_t stream);

/* The input gradient's two shares (bf16 layers):
 *   dx[t] = sum_e dlogits[t, e] W_router[e]  +  sum_{j<k} dxd[tok_row[t, j]]  (+ dxd[R + t])
 * accumulated in fp32 and written once in bf16; on the tensor-core path (below) the
 * router's share is first rounded to bf16 and added last. dxd = NULL leaves the dispatch
 * share out (dx = the router's share alone; tok_row is then not read). tok_row is the
 * forward's map, trusted as in moe_dispatch_backward. H % 8 == 0. ws:
 * moe_router_backward_workspace_size bytes, initialised with moe_workspace_init.
 *
 * Precision of the router's products: with E % 128 == 0, H % 256 == 0 and bf16 layers
 * (and k + shared <= 9), dw_router = dl^T x and dl W_router run on the tensor cores with
 * dlogits rounded to bf16 and fp32 accumulation, as the expert GEMMs do; dlogits itself
 * stays fp32. Otherwise both are fp32 FMA products. */
moe_status_t moe_dispatch_router_backward(const moe_config_t* cfg, const void* dxd, const int32_t* tok_row,
                                          const float* dlogits, const void* w_router, void* dx, void* ws,
                                          moe_stream_t stream);

/* Offline weight preparation for the E4M3 variant: quantise a bf16 [rows, cols] matrix in
 * br x bc blocks with the rule of moe_dispatch; q [rows, cols] e4m3, scale
 * [ceil(rows/br), ceil(cols/bc)] fp32 row-major. br, bc in {1, 128}. */
moe_status_t moe_quantize_e4m3(const void* src_bf16, int64_t rows, int64_t cols, int32_t br,
                               int32_t bc, uint8_t* q, float* scale, moe_stream_t stream);

/* Offline weight preparation for the MXFP8 variant: quantise a bf16 [rows, cols] matrix
 * along its rows in 1x32 blocks with the rule of moe_dispatch_mx; q [rows, cols] e4m3, sf
 * the scale atoms with tile a = rows [128a, 128a + 128): (rows/128) * (cols/128) * 512
 * bytes. rows % 128 == 0 and cols % 128 == 0 (else MOE_ERR_UNSUPPORTED). For the expert
 * weights pass [E*F, H] (gate, up) and [E*H, F] (down). */
moe_status_t moe_quantize_mx(const void* src_bf16, int64_t rows, int64_t cols, uint8_t* q,
                             uint8_t* sf, moe_stream_t stream);

/* moe_route for callers that cannot allocate device memory. The paper has no counterpart:
 * this is a library convenience. It computes exactly what moe_route computes (the same
 * per-token routing code and the same map, bit for bit; here a top-k launch and the scan
 * passes instead of moe_route's single cooperative launch) but takes no workspace: the routing scan's scratch lives in a fixed array
 * inside the library (1 MiB of device memory per GPU that loads the library, held until
 * the process exits). It is meant for callers that are handed only their inputs and
 * outputs (a plugin inside a host framework), that run on a fixed memory budget reserved
 * up front, or that run where allocating is not allowed (an allocator's own callback).
 *  - Limit: ceil(T / 128) * E <= 262144 (e.g. T = 131072 tokens with E = 256); larger
 *    problems return MOE_ERR_UNSUPPORTED before anything is launched.
 *  - A call looks up the array's device address (no allocation) when the device's current
 *    context is not the one it last looked it up in: the first call on each device, and the
 *    first call after the device was reset. Make such a first call before any stream
 *    capture.
 *  - Every call on a device shares the one array: calls whose kernels overlap on the GPU
 *    (two streams, two host threads) race, and the caller must serialise them.
 *  - device_status: optional caller-owned device int32[2] (code, detail) that receives
 *    device-detected faults (non-finite scores) like the workspace's status word; zero it
 *    before the call. With NULL those faults are not reported (outputs stay in bounds).
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. */
moe_status_t moe_route_static_scratch(const moe_config_t* cfg, const float* logits,
                                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                                      int32_t* offsets, int32_t* row_token, int32_t* tok_row,
                                      int32_t* device_status, moe_stream_t stream);

/* Diagnostic: runs the bounded wait that guards every wait inside the library's tensor-core
 * kernels on a barrier nothing arrives on. With a working limit it records MOE_ERR_TIMEOUT
 * in device_status (caller-owned device int32[2], zeroed by the caller) after about
 * timeout_ns (0 < timeout_ns <= 10 s) and returns, and the context stays usable. */
moe_status_t moe_selftest_bounded_wait(int64_t timeout_ns, int32_t* device_status,
                                       moe_stream_t stream);

/* Synchronises `stream`, returns the device status word of `ws` in *device_status
 * (MOE_OK or a moe_status_t code) and clears it. The only call that blocks the host. */
moe_status_t moe_read_status(void* ws, moe_stream_t stream, int32_t* device_status);

/* Static string naming a status code. */
const char* moe_status_string(moe_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
