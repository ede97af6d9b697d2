// The C ABI (include/moe.h): host-side validation, workspace layout and the stream-ordered
// sequence of kernels. Nothing here synchronises the host except moe_read_status, and
// nothing allocates device memory: every buffer is the caller's.
#include <string.h>

#include "moe_internal.cuh"
#include "gemm_tc.cuh"
#include "mx_common.cuh"

using namespace moe;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool ptr_ok(const void* p) { return p != nullptr && aligned16(p); }

moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H <= 0 || c->E < 1 || c->k < 1 || c->F <= 0) return MOE_ERR_INVALID_ARG;
  if (c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->k > 32 || c->E > 512) return MOE_ERR_UNSUPPORTED;
  if (c->n_groups < 1 || c->E % c->n_groups != 0) return MOE_ERR_INVALID_ARG;
  if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 32) return MOE_ERR_UNSUPPORTED;
  if (c->score_fn != MOE_SCORE_SOFTMAX && c->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->group_score != MOE_GROUP_SCORE_TOP2_SUM && c->group_score != MOE_GROUP_SCORE_MAX) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 1 && c->topk_groups < c->n_groups) {
    if (c->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)c->topk_groups * (c->E / c->n_groups) < c->k) return MOE_ERR_INVALID_ARG;
  }
  if (c->act_dtype != MOE_DTYPE_F32 && c->act_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  const bool quant = c->xfer_dtype == MOE_DTYPE_E4M3 || c->xfer_dtype == MOE_DTYPE_MXE4M3;
  if (c->xfer_dtype != c->act_dtype && !quant) return MOE_ERR_INVALID_ARG;
  if (quant && c->act_dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_UNSUPPORTED;
  if (c->n_shared && c->F_shared != c->F) return MOE_ERR_UNSUPPORTED;
  // rows move as 8-element (16-byte bf16) steps in dispatch and combine
  if (c->H % 8 || c->F % 8) return MOE_ERR_UNSUPPORTED;
  if (quant && (c->H % 128 || c->F % 128)) return MOE_ERR_UNSUPPORTED;
  if (total_rows(*c) >= (int64_t)INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// T = 0: nothing routed; counts and offsets (if given) become zero.
moe_status_t empty_routing(const moe_config_t& c, int32_t* counts, int32_t* offsets, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (counts && aligned16(counts)) e = cudaMemsetAsync(counts, 0, (size_t)c.E * 4, s);
  if (e == cudaSuccess && offsets && aligned16(offsets)) e = cudaMemsetAsync(offsets, 0, (size_t)(c.E + 1) * 4, s);
  return cuda_status(e);
}

// Workspace head: the status word at byte 0, the fused routing kernel's grid barrier
// (counter, flag) at byte 16; then the routing scratch (per-block expert counts).
DeviceStatus* status_of(void* ws) { return reinterpret_cast<DeviceStatus*>(ws); }
uint32_t* barrier_of(void* ws) { return reinterpret_cast<uint32_t*>((char*)ws + 128); }
int32_t* blockcnt_of(void* ws) { return reinterpret_cast<int32_t*>((char*)ws + kWsHead); }

// The routing workspace: the head, the scan's (or the single launch's) per-block counts, and
// the auxiliary loss's per-block 64-bit partial sums.
size_t route_blocks(const moe_config_t& c) {
  return std::max<size_t>((size_t)scan_blocks(c), (size_t)kFusedMaxRouteBlocks);
}
uint64_t* auxp_of(void* ws, const moe_config_t& c) {
  return reinterpret_cast<uint64_t*>((char*)ws + kWsHead + align_up(route_blocks(c) * c.E * sizeof(int32_t), 256));
}
size_t route_ws_bytes(const moe_config_t& c) {
  return kWsHead + align_up(route_blocks(c) * c.E * sizeof(int32_t), 256) +
         align_up(route_blocks(c) * c.E * sizeof(uint64_t), 256);
}

// S1 + S2: one cooperative launch where it applies, else the top-k and scan passes.
// S1 + S2, and with aux_loss the auxiliary loss: inside the single routing launch where there
// is one, else by its own two launches after the scan.
cudaError_t route_and_permute(const moe_config_t& c, const float* logits, int32_t* topk_idx, float* topk_w,
                              int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* tok_row, void* ws,
                              cudaStream_t s, float aux_alpha = 0.0f, float* aux_loss = nullptr) {
  if (route_fused_supported(c))
    return launch_route_fused(c, logits, topk_idx, topk_w, counts, offsets, row_token, tok_row, blockcnt_of(ws),
                              barrier_of(ws), status_of(ws), s, aux_loss ? auxp_of(ws, c) : nullptr, aux_alpha,
                              aux_loss);
  cudaError_t e = launch_route_topk(c, logits, topk_idx, topk_w, status_of(ws), s);
  if (e == cudaSuccess)
    e = launch_route_scan(c, topk_idx, counts, offsets, row_token, tok_row, blockcnt_of(ws), status_of(ws), s);
  if (e == cudaSuccess && aux_loss) e = launch_aux_loss(c, logits, counts, aux_alpha, aux_loss, auxp_of(ws, c), s);
  return e;
}

size_t act_size(const moe_config_t& c) { return c.act_dtype == MOE_DTYPE_BF16 ? 2 : 4; }
bool is_mx(const moe_config_t& c) { return c.xfer_dtype == MOE_DTYPE_MXE4M3; }
bool is_quant(const moe_config_t& c) { return c.xfer_dtype == MOE_DTYPE_E4M3 || is_mx(c); }
size_t xfer_size(const moe_config_t& c) { return is_quant(c) ? 1 : act_size(c); }

// Bytes of the scales of the grouped activations with K columns.
size_t act_scale_bytes(const moe_config_t& c, int K) {
  if (c.xfer_dtype == MOE_DTYPE_E4M3) return (size_t)total_rows(c) * (K / 128) * 4;
  if (is_mx(c)) return (size_t)mx_act_atom_rows(c) * (K / 128) * 512;
  return 0;
}

// Layers the gathered-row GEMM1 (moe_grouped_mlp_gather) takes: bf16 on the tensor cores.
// moe_forward does not use it: on GB300 the 32 four-row TMA gathers per K block cost more
// than the separate dispatch pass they save (measured by bench.py as grouped_mlp_gather).
bool fused_gather(const moe_config_t& c) {
  return c.act_dtype == MOE_DTYPE_BF16 && c.xfer_dtype == MOE_DTYPE_BF16 && tc::mlp_supported(c);
}

// moe_forward's workspace: the routing part, then every intermediate.
struct FwdLayout {
  size_t logits, topk_idx, topk_w, counts, offsets, row_token, tok_row, xd, xd_scale, h, h_scale,
      yd, total;
};

FwdLayout fwd_layout(const moe_config_t& c) {
  FwdLayout L;
  size_t o = route_ws_bytes(c);
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const int64_t Tk = (int64_t)c.T * c.k, rows = total_rows(c);
  L.logits = take((size_t)c.T * c.E * 4);
  L.topk_idx = take((size_t)Tk * 4);
  L.topk_w = take((size_t)Tk * 4);
  L.counts = take((size_t)c.E * 4);
  L.offsets = take((size_t)(c.E + 1) * 4);
  L.row_token = take((size_t)Tk * 4);
  L.tok_row = take((size_t)Tk * 4);
  L.xd = take((size_t)rows * c.H * xfer_size(c));
  L.xd_scale = take(act_scale_bytes(c, c.H));
  L.h = take((size_t)rows * c.F * xfer_size(c));
  L.h_scale = take(act_scale_bytes(c, c.F));
  L.yd = take((size_t)rows * c.H * act_size(c));
  L.total = o;
  return L;
}

// Backward workspace: status head, then dyd, dxd [rows, H], gu [rows, 2F], dgu [prows, 2F],
// h [prows, F] (prows: every expert's rows padded to a multiple of 64), then the router's
// dlogits [T, E] and its weight gradient's per-slice partial sums [S, E, H] and [S, E].
struct BwdLayout {
  size_t dyd, dxd, gu, dgu, h, dl, rpart, rbpart, dlb, dxr, roff, total;
};

// Router backward partial sums: the SIMT path's token slices, or the tensor-core path's.
size_t router_part_slices(const moe_config_t& c) {
  if (!router_backward_tc(c)) return (size_t)router_wgrad_slices(c);
  int slice, slices;
  router_tc_slices(c, &slice, &slices);
  return slices > 1 ? (size_t)slices : 0;
}

BwdLayout bwd_layout(const moe_config_t& c) {
  BwdLayout L;
  size_t o = kWsHead;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t rows = (size_t)total_rows(c);
  const size_t prows = (size_t)tc::backward_padded_rows(c);  // dgu and h: 64-row padded segments
  const size_t S = (size_t)router_wgrad_slices(c);
  L.dyd = take(rows * c.H * 2);
  L.dxd = take(rows * c.H * 2);
  L.gu = take(rows * 2 * c.F * 2);
  L.dgu = take(prows * 2 * c.F * 2);
  L.h = take(prows * c.F * 2);
  const bool tcr = router_backward_tc(c);
  L.dl = take((size_t)c.T * c.E * 4);
  L.rpart = take(router_part_slices(c) * c.E * c.H * 4);
  L.rbpart = take(std::max(S, (size_t)router_bias_slices(c)) * c.E * 4);
  L.dlb = take(tcr ? (size_t)c.T * c.E * 2 : 0);
  L.dxr = take(tcr ? (size_t)c.T * c.H * 2 : 0);
  L.roff = take(256 * 4);
  L.total = o;
  return L;
}

// moe_router_backward's and moe_dispatch_router_backward's workspace: status head, then the
// partial sums of the SIMT path, or dl in bf16 and dx_r on the tensor-core path.
struct RouterBwdLayout {
  size_t rpart, rbpart, dlb, dxr, roff, total;
};

RouterBwdLayout router_bwd_layout(const moe_config_t& c) {
  RouterBwdLayout L;
  size_t o = kWsHead;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t S = (size_t)router_wgrad_slices(c);
  const bool tcr = router_backward_tc(c);
  L.rpart = take(router_part_slices(c) * c.E * c.H * 4);
  L.rbpart = take(std::max(S, (size_t)router_bias_slices(c)) * c.E * 4);
  L.dlb = take(tcr ? (size_t)c.T * c.E * 2 : 0);
  L.dxr = take(tcr ? (size_t)c.T * c.H * 2 : 0);
  L.roff = take(256 * 4);
  L.total = o;
  return L;
}

RouterScratch router_scratch(char* base, size_t part, size_t bias_part, size_t dlb, size_t dxr, size_t roff) {
  return RouterScratch{reinterpret_cast<float*>(base + part), reinterpret_cast<float*>(base + bias_part), base + dlb,
                       base + dxr, reinterpret_cast<int32_t*>(base + roff)};
}

bool opt_ok(const void* p) { return p == nullptr || aligned16(p); }

bool grads_ok(const moe_config_t& c, const moe_weight_grads_t* g) {
  if (!g || !ptr_ok(g->dw_gate) || !ptr_ok(g->dw_up) || !ptr_ok(g->dw_down)) return false;
  if (c.n_shared && (!ptr_ok(g->dws_gate) || !ptr_ok(g->dws_up) || !ptr_ok(g->dws_down))) return false;
  if (!opt_ok(g->dw_router) || !opt_ok(g->d_router_bias) || !opt_ok(g->dlogits)) return false;
  if (!g->dw_router && g->d_router_bias) return false;  // the bias gradient comes with the weight's
  if (!(g->aux_loss_coeff == g->aux_loss_coeff)) return false;  // NaN
  return true;
}

moe_status_t check_weights(const moe_config_t& c, const moe_weights_t* w, bool need_router) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (need_router && !ptr_ok(w->w_router)) return MOE_ERR_INVALID_ARG;
  if (w->router_bias && !aligned16(w->router_bias)) return MOE_ERR_INVALID_ARG;
  if (!ptr_ok(w->w_gate) || !ptr_ok(w->w_up) || !ptr_ok(w->w_down)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = is_quant(c);
  if (fp8 && (!ptr_ok(w->s_gate) || !ptr_ok(w->s_up) || !ptr_ok(w->s_down))) return MOE_ERR_INVALID_ARG;
  if (c.n_shared) {
    if (!ptr_ok(w->ws_gate) || !ptr_ok(w->ws_up) || !ptr_ok(w->ws_down)) return MOE_ERR_INVALID_ARG;
    if (fp8 && (!ptr_ok(w->ss_gate) || !ptr_ok(w->ss_up) || !ptr_ok(w->ss_down))) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

cudaError_t router_logits(const moe_config_t& c, const void* x, const void* w_router,
                          const float* bias, float* logits, DeviceStatus* st, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (c.act_dtype == MOE_DTYPE_BF16 && tc::router_supported(c))
    return tc::launch_router(c, x, w_router, bias, logits, st, s);
  if (router_small_supported(c)) return launch_router_small(c, x, w_router, bias, logits, s);
  SimtGemmArgs a{};
  a.mode = 0;
  a.act_bf16 = c.act_dtype == MOE_DTYPE_BF16;
  a.M_static = c.T;
  a.A = x;
  a.B0 = w_router;
  a.bias = bias;
  a.C = logits;
  a.N = c.E;
  a.K = c.H;
  return launch_simt_gemm(a, s);
}

cudaError_t grouped_mlp(const moe_config_t& c, const void* xd, const void* xd_scale,
                        const void* x, const int32_t* offsets, const moe_weights_t& w, void* h,
                        void* h_scale, void* yd, DeviceStatus* st, cudaStream_t s) {
  if (c.T == 0) return cudaSuccess;
  if (is_mx(c)) return tc::launch_grouped_mlp_mx(c, xd, xd_scale, offsets, w, h, h_scale, yd, st, s);
  if (tc::mlp_supported(c))
    return tc::launch_grouped_mlp(c, xd, static_cast<const float*>(xd_scale), x, offsets, w, h,
                                  static_cast<float*>(h_scale), yd, st, s);
  // exact-fp32 FFMA path (fp32 layers, and bf16 shapes the tensor-core tiles do not take)
  const int64_t R = routed_rows(c);
  SimtGemmArgs a{};
  a.act_bf16 = c.act_dtype == MOE_DTYPE_BF16;
  a.M_static = -1;
  a.offsets = offsets;
  a.G = c.E;
  a.extra_group = c.n_shared ? 1 : 0;
  a.routed_rows = R;
  a.T_extra = c.T;
  // gate/up: h = silu(xd Wg^T) * (xd Wu^T)
  a.mode = 1;
  a.A = xd;
  a.A_extra = x;
  a.B0 = w.w_gate;
  a.B1 = w.w_up;
  a.B0_extra = w.ws_gate;
  a.B1_extra = w.ws_up;
  a.C = h;
  a.N = c.F;
  a.K = c.H;
  cudaError_t e = launch_simt_gemm(a, s);
  if (e != cudaSuccess) return e;
  // down: yd = h Wd^T
  a.mode = 2;
  a.A = h;
  a.A_extra = (const char*)h + (size_t)R * c.F * act_size(c);
  a.B0 = w.w_down;
  a.B1 = nullptr;
  a.B0_extra = w.ws_down;
  a.B1_extra = nullptr;
  a.C = yd;
  a.N = c.H;
  a.K = c.F;
  return launch_simt_gemm(a, s);
}

}  // namespace

extern "C" {

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = route_ws_bytes(*cfg);
  return MOE_OK;
}

moe_status_t moe_forward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = fwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_workspace_init(void* ws, moe_stream_t stream) {
  if (!ptr_ok(ws)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, kWsHead, (cudaStream_t)stream));
}

moe_status_t moe_router_logits(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, float* logits, void* ws,
                               moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(x) || !ptr_ok(w_router) || !ptr_ok(logits) || !ptr_ok(ws)) return MOE_ERR_INVALID_ARG;
  if (router_bias && !aligned16(router_bias)) return MOE_ERR_INVALID_ARG;
  return cuda_status(router_logits(*cfg, x, w_router, router_bias, logits, status_of(ws),
                                   (cudaStream_t)stream));
}

moe_status_t moe_route(const moe_config_t* cfg, const float* logits, int32_t* topk_idx,
                       float* topk_w, int32_t* counts, int32_t* offsets, int32_t* row_token,
                       int32_t* tok_row, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return empty_routing(*cfg, counts, offsets, (cudaStream_t)stream);
  if (!ptr_ok(logits) || !ptr_ok(topk_idx) || !ptr_ok(topk_w) || !ptr_ok(counts) ||
      !ptr_ok(offsets) || !ptr_ok(row_token) || !ptr_ok(tok_row) || !ptr_ok(ws))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(route_and_permute(*cfg, logits, topk_idx, topk_w, counts, offsets, row_token, tok_row, ws,
                                       (cudaStream_t)stream));
}

moe_status_t moe_route_launch_count(const moe_config_t* cfg, int32_t* launches) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!launches) return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = *cfg;
  *launches = c.T == 0 ? 0 : route_fused_supported(c) ? 1 : (c.T <= 512 ? 2 : 4);
  return MOE_OK;
}

moe_status_t moe_route_from_map(const moe_config_t* cfg, const int32_t* topk_idx,
                                int32_t* counts, int32_t* offsets, int32_t* row_token,
                                int32_t* tok_row, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return empty_routing(*cfg, counts, offsets, (cudaStream_t)stream);
  if (!ptr_ok(topk_idx) || !ptr_ok(counts) || !ptr_ok(offsets) || !ptr_ok(row_token) ||
      !ptr_ok(tok_row) || !ptr_ok(ws))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_route_scan(*cfg, topk_idx, counts, offsets, row_token, tok_row,
                                       blockcnt_of(ws), status_of(ws), (cudaStream_t)stream));
}

moe_status_t moe_aux_loss(const moe_config_t* cfg, const float* logits, const int32_t* counts,
                          float alpha, float* loss, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!ptr_ok(counts) || !loss || !ptr_ok(ws) || (cfg->T > 0 && !ptr_ok(logits))) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_aux_loss(*cfg, logits, counts, alpha, loss, auxp_of(ws, *cfg), (cudaStream_t)stream));
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* tok_row,
                          void* xd, float* xd_scale, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(x) || !ptr_ok(tok_row) || !ptr_ok(xd)) return MOE_ERR_INVALID_ARG;
  if (is_mx(*cfg)) return MOE_ERR_UNSUPPORTED;  // moe_dispatch_mx
  if (cfg->xfer_dtype == MOE_DTYPE_E4M3 && !ptr_ok(xd_scale)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch(*cfg, x, tok_row, xd, xd_scale, (cudaStream_t)stream));
}

moe_status_t moe_dispatch_mx(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                             const int32_t* tok_row, const int32_t* offsets, void* xd, void* xd_sf,
                             moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!is_mx(*cfg)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(x) || !ptr_ok(topk_idx) || !ptr_ok(tok_row) || !ptr_ok(offsets) || !ptr_ok(xd) || !ptr_ok(xd_sf))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch_mx(*cfg, x, topk_idx, tok_row, offsets, xd, xd_sf, (cudaStream_t)stream));
}

moe_status_t moe_mx_scale_bytes(const moe_config_t* cfg, int32_t K, size_t* bytes) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!bytes || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 128) return MOE_ERR_UNSUPPORTED;
  *bytes = (size_t)mx_act_atom_rows(*cfg) * (K / 128) * 512;
  return MOE_OK;
}

moe_status_t moe_grouped_mlp(const moe_config_t* cfg, const void* xd, const void* xd_scale,
                             const void* x, const int32_t* offsets, const moe_weights_t* w,
                             void* h, void* h_scale, void* yd, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return MOE_OK;
  v = check_weights(*cfg, w, false);
  if (v != MOE_OK) return v;
  const bool fp8 = is_quant(*cfg);
  if (!ptr_ok(xd) || !ptr_ok(offsets) || !ptr_ok(h) || !ptr_ok(yd) || !ptr_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (fp8 && (!ptr_ok(xd_scale) || !ptr_ok(h_scale))) return MOE_ERR_INVALID_ARG;
  if (cfg->n_shared && !fp8 && !ptr_ok(x)) return MOE_ERR_INVALID_ARG;
  if (fp8 && !tc::mlp_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(grouped_mlp(*cfg, xd, xd_scale, x, offsets, *w, h, h_scale, yd,
                                 status_of(ws), (cudaStream_t)stream));
}

moe_status_t moe_grouped_mlp_gather(const moe_config_t* cfg, const void* x, const int32_t* row_token,
                                    const int32_t* offsets, const int32_t* tok_row, const float* topk_w,
                                    const moe_weights_t* w, void* h, void* yd, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if ((tok_row == nullptr) != (topk_w == nullptr)) return MOE_ERR_INVALID_ARG;  // both or neither
  if (cfg->T == 0) return MOE_OK;
  v = check_weights(*cfg, w, false);
  if (v != MOE_OK) return v;
  if (!ptr_ok(x) || !ptr_ok(row_token) || !ptr_ok(offsets) || !ptr_ok(h) || !ptr_ok(yd) || !ptr_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (!fused_gather(*cfg)) return MOE_ERR_UNSUPPORTED;
  return cuda_status(tc::launch_grouped_mlp(*cfg, nullptr, nullptr, x, offsets, *w, h, nullptr, yd, status_of(ws),
                                            (cudaStream_t)stream, row_token, tok_row, topk_w));
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* yd, const int32_t* tok_row,
                         const float* topk_w, void* y, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->T == 0) return MOE_OK;
  // topk_w NULL: unit weights (rows already weighted by moe_grouped_mlp_gather)
  if (!ptr_ok(yd) || !ptr_ok(tok_row) || (topk_w != nullptr && !ptr_ok(topk_w)) || !ptr_ok(y))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, yd, tok_row, topk_w, y, (cudaStream_t)stream));
}

namespace {
// moe_forward, and with keep (moe_forward_train) GEMM1 also keeps g and u in gu_keep.
moe_status_t forward_impl(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y, void* ws,
                          int32_t* topk_idx_out, float* topk_w_out, int32_t* counts_out, bool keep, void* gu_keep,
                          moe_stream_t stream, float aux_alpha = 0.0f, float* aux_loss_out = nullptr) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (keep && !tc::mlp_backward_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (aux_loss_out && !(aux_alpha == aux_alpha)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0)
    return aux_loss_out ? cuda_status(cudaMemsetAsync(aux_loss_out, 0, sizeof(float), (cudaStream_t)stream)) : MOE_OK;
  v = check_weights(*cfg, w, true);
  if (v != MOE_OK) return v;
  if (!ptr_ok(x) || !ptr_ok(y) || !ptr_ok(ws) || (keep && !ptr_ok(gu_keep))) return MOE_ERR_INVALID_ARG;
  if ((topk_idx_out && !aligned16(topk_idx_out)) || (topk_w_out && !aligned16(topk_w_out)) ||
      (counts_out && !aligned16(counts_out)))
    return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = *cfg;
  if (is_quant(c) && !tc::mlp_supported(c)) return MOE_ERR_UNSUPPORTED;
  if (c.T == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const FwdLayout L = fwd_layout(c);
  char* base = (char*)ws;
  float* logits = (float*)(base + L.logits);
  int32_t* topk_idx = (int32_t*)(base + L.topk_idx);
  float* topk_w = (float*)(base + L.topk_w);
  int32_t* counts = (int32_t*)(base + L.counts);
  int32_t* offsets = (int32_t*)(base + L.offsets);
  int32_t* row_token = (int32_t*)(base + L.row_token);
  int32_t* tok_row = (int32_t*)(base + L.tok_row);
  void* xd = base + L.xd;
  void* xd_scale = is_quant(c) ? (void*)(base + L.xd_scale) : nullptr;
  void* h = base + L.h;
  void* h_scale = is_quant(c) ? (void*)(base + L.h_scale) : nullptr;
  void* yd = base + L.yd;

  cudaError_t e = router_logits(c, x, w->w_router, w->router_bias, logits, status_of(ws), s);
  if (e == cudaSuccess)
    e = route_and_permute(c, logits, topk_idx, topk_w, counts, offsets, row_token, tok_row, ws, s, aux_alpha,
                          aux_loss_out);
  if (e == cudaSuccess)
    e = is_mx(c) ? launch_dispatch_mx(c, x, topk_idx, tok_row, offsets, xd, xd_scale, s)
                 : launch_dispatch(c, x, tok_row, xd, static_cast<float*>(xd_scale), s);
  if (e == cudaSuccess)
    e = keep ? tc::launch_grouped_mlp(c, xd, nullptr, x, offsets, *w, h, nullptr, yd, status_of(ws), s, nullptr,
                                         nullptr, nullptr, gu_keep)
                : grouped_mlp(c, xd, xd_scale, x, offsets, *w, h, h_scale, yd, status_of(ws), s);
  if (e == cudaSuccess) e = launch_combine(c, yd, tok_row, topk_w, y, s);
  const size_t Tk = (size_t)c.T * c.k;
  if (e == cudaSuccess && topk_idx_out)
    e = cudaMemcpyAsync(topk_idx_out, topk_idx, Tk * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && topk_w_out)
    e = cudaMemcpyAsync(topk_w_out, topk_w, Tk * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && counts_out)
    e = cudaMemcpyAsync(counts_out, counts, (size_t)c.E * 4, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}
}  // namespace

moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const moe_weights_t* w,
                         void* y, void* ws, int32_t* topk_idx_out, float* topk_w_out,
                         int32_t* counts_out, moe_stream_t stream) {
  return forward_impl(cfg, x, w, y, ws, topk_idx_out, topk_w_out, counts_out, false, nullptr, stream);
}

moe_status_t moe_forward_train(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y, void* ws,
                               void* gu, float aux_alpha, float* aux_loss, moe_stream_t stream) {
  return forward_impl(cfg, x, w, y, ws, nullptr, nullptr, nullptr, true, gu, stream, aux_alpha, aux_loss);
}

moe_status_t moe_forward_host(const moe_config_t* cfg, const void* x_host, const moe_weights_t* w,
                              void* y_host, void* x_dev, void* y_dev, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (x_host == nullptr || y_host == nullptr || !ptr_ok(x_dev) || !ptr_ok(y_dev)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  const size_t bytes = (size_t)cfg->T * cfg->H * act_size(*cfg);
  cudaStream_t s = (cudaStream_t)stream;
  v = cuda_status(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s));
  if (v != MOE_OK) return v;
  v = moe_forward(cfg, x_dev, w, y_dev, ws, nullptr, nullptr, nullptr, stream);
  if (v != MOE_OK) return v;
  return cuda_status(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, s));
}

moe_status_t moe_quantize_e4m3(const void* src_bf16, int64_t rows, int64_t cols, int32_t br,
                               int32_t bc, uint8_t* q, float* scale, moe_stream_t stream) {
  if (!ptr_ok(src_bf16) || !ptr_ok(q) || !ptr_ok(scale) || rows < 0 || cols < 0)
    return MOE_ERR_INVALID_ARG;
  if ((br != 1 && br != 128) || (bc != 1 && bc != 128)) return MOE_ERR_UNSUPPORTED;
  if (ceil_div(rows, br) * ceil_div(cols, bc) > (int64_t)INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_quantize_e4m3(src_bf16, rows, cols, br, bc, q, scale, (cudaStream_t)stream));
}

moe_status_t moe_backward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (!tc::mlp_backward_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  *bytes = bwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_combine_backward(const moe_config_t* cfg, const void* dy, const void* yd, const int32_t* tok_row,
                                  const float* topk_w, void* dyd, float* dtopk_w, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->act_dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(dy) || !ptr_ok(yd) || !ptr_ok(tok_row) || !ptr_ok(topk_w) || !ptr_ok(dyd) || !ptr_ok(dtopk_w))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_backward(*cfg, dy, yd, tok_row, topk_w, dyd, dtopk_w, (cudaStream_t)stream));
}

moe_status_t moe_grouped_mlp_backward(const moe_config_t* cfg, const void* xd, const void* x, const int32_t* offsets,
                                      const moe_weights_t* w, const void* dyd, void* dxd,
                                      const moe_weight_grads_t* grads, void* ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!tc::mlp_backward_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  v = check_weights(*cfg, w, false);
  if (v != MOE_OK) return v;
  if (!grads_ok(*cfg, grads)) return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = *cfg;
  cudaStream_t s = (cudaStream_t)stream;
  if (c.T > 0 && (!ptr_ok(xd) || !ptr_ok(offsets) || !ptr_ok(dyd) || !ptr_ok(dxd) || !ptr_ok(ws) ||
                  (c.n_shared && !ptr_ok(x))))
    return MOE_ERR_INVALID_ARG;
  if (c.T == 0) {  // no rows: every weight gradient is zero
    cudaError_t e = cudaMemsetAsync(grads->dw_gate, 0, (size_t)c.E * c.F * c.H * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(grads->dw_up, 0, (size_t)c.E * c.F * c.H * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(grads->dw_down, 0, (size_t)c.E * c.F * c.H * 4, s);
    if (e == cudaSuccess && c.n_shared) e = cudaMemsetAsync(grads->dws_gate, 0, (size_t)c.F * c.H * 4, s);
    if (e == cudaSuccess && c.n_shared) e = cudaMemsetAsync(grads->dws_up, 0, (size_t)c.F * c.H * 4, s);
    if (e == cudaSuccess && c.n_shared) e = cudaMemsetAsync(grads->dws_down, 0, (size_t)c.F * c.H * 4, s);
    return cuda_status(e);
  }
  const BwdLayout L = bwd_layout(c);
  char* base = (char*)ws;
  return cuda_status(tc::launch_grouped_mlp_backward(c, xd, x, offsets, *w, dyd, base + L.gu, base + L.dgu,
                                                     base + L.h, dxd, *grads, status_of(ws), s));
}

moe_status_t moe_dispatch_backward(const moe_config_t* cfg, const void* dxd, const int32_t* tok_row, void* dx,
                                   moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->act_dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(dxd) || !ptr_ok(tok_row) || !ptr_ok(dx)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*cfg, dxd, tok_row, nullptr, dx, (cudaStream_t)stream));
}

namespace {
moe_status_t backward_impl(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                           const void* fwd_ws, const void* gu_kept, void* dx, float* dtopk_w,
                           const moe_weight_grads_t* grads, void* bwd_ws, moe_stream_t stream);
}  // namespace

moe_status_t moe_backward(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                          const void* fwd_ws, void* dx, float* dtopk_w, const moe_weight_grads_t* grads, void* bwd_ws,
                          moe_stream_t stream) {
  return backward_impl(cfg, x, w, dy, fwd_ws, nullptr, dx, dtopk_w, grads, bwd_ws, stream);
}

moe_status_t moe_backward_kept(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                               const void* fwd_ws, const void* gu, void* dx, float* dtopk_w,
                               const moe_weight_grads_t* grads, void* bwd_ws, moe_stream_t stream) {
  if (cfg && cfg->T > 0 && !ptr_ok(gu)) return MOE_ERR_INVALID_ARG;  // (T = 0 reads nothing)
  return backward_impl(cfg, x, w, dy, fwd_ws, gu, dx, dtopk_w, grads, bwd_ws, stream);
}

namespace {
moe_status_t backward_impl(const moe_config_t* cfg, const void* x, const moe_weights_t* w, const void* dy,
                           const void* fwd_ws, const void* gu_kept, void* dx, float* dtopk_w,
                           const moe_weight_grads_t* grads, void* bwd_ws, moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!tc::mlp_backward_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) {
    v = moe_grouped_mlp_backward(cfg, nullptr, nullptr, nullptr, w, nullptr, nullptr, grads, bwd_ws, stream);
    if (v != MOE_OK || !grads->dw_router) return v;
    return cuda_status(launch_router_backward(*cfg, nullptr, nullptr, nullptr, nullptr, 0.0f, nullptr, nullptr,
                                              grads->dw_router, grads->d_router_bias, RouterScratch{},
                                              nullptr, (cudaStream_t)stream));
  }
  v = check_weights(*cfg, w, false);
  if (v != MOE_OK) return v;
  if (!ptr_ok(x) || !ptr_ok(dy) || !ptr_ok(fwd_ws) || !ptr_ok(dx) || !ptr_ok(dtopk_w) || !ptr_ok(bwd_ws) ||
      !grads_ok(*cfg, grads))
    return MOE_ERR_INVALID_ARG;
  if (grads->dw_router && cfg->H % 8) return MOE_ERR_UNSUPPORTED;
  const moe_config_t& c = *cfg;
  cudaStream_t s = (cudaStream_t)stream;
  const FwdLayout F = fwd_layout(c);
  const BwdLayout B = bwd_layout(c);
  const char* fb = (const char*)fwd_ws;
  char* bb = (char*)bwd_ws;
  const int32_t* tok_row = (const int32_t*)(fb + F.tok_row);
  cudaError_t e = launch_combine_backward(c, dy, fb + F.yd, tok_row, (const float*)(fb + F.topk_w), bb + B.dyd,
                                          dtopk_w, s);
  if (e == cudaSuccess)
    e = tc::launch_grouped_mlp_backward(c, fb + F.xd, x, (const int32_t*)(fb + F.offsets), *w, bb + B.dyd,
                                        gu_kept ? const_cast<void*>(gu_kept) : (void*)(bb + B.gu), bb + B.dgu,
                                        bb + B.h, bb + B.dxd, *grads, status_of(bwd_ws), s, gu_kept != nullptr);
  if (!grads->dw_router) {
    if (e == cudaSuccess) e = launch_combine(c, bb + B.dxd, tok_row, nullptr, dx, s);
    return cuda_status(e);
  }
  float* dl = grads->dlogits ? grads->dlogits : (float*)(bb + B.dl);
  const int32_t* counts = grads->aux_loss_coeff != 0.0f ? (const int32_t*)(fb + F.counts) : nullptr;
  const RouterScratch sc = router_scratch(bb, B.rpart, B.rbpart, B.dlb, B.dxr, B.roff);
  if (e == cudaSuccess)
    e = launch_router_backward(c, (const float*)(fb + F.logits), (const int32_t*)(fb + F.topk_idx), dtopk_w, counts,
                               grads->aux_loss_coeff, x, dl, grads->dw_router, grads->d_router_bias, sc,
                               status_of(bwd_ws), s);
  if (e == cudaSuccess)
    e = launch_router_input_grad(c, dl, router_backward_tc(c) ? sc.dl_bf16 : nullptr, w->w_router, bb + B.dxd,
                                 tok_row, dx, sc, status_of(bwd_ws), s);
  return cuda_status(e);
}

}  // namespace

moe_status_t moe_router_backward_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = router_bwd_layout(*cfg).total;
  return MOE_OK;
}

moe_status_t moe_router_backward(const moe_config_t* cfg, const float* logits, const int32_t* topk_idx,
                                 const float* dtopk_w, const int32_t* counts, float aux_alpha, const void* x,
                                 float* dlogits, float* dw_router, float* d_router_bias, void* ws,
                                 moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->H % 8) return MOE_ERR_UNSUPPORTED;
  if (!opt_ok(counts) || !opt_ok(dw_router) || !opt_ok(d_router_bias) || !(aux_alpha == aux_alpha) ||
      (!dw_router && d_router_bias))
    return MOE_ERR_INVALID_ARG;
  const moe_config_t& c = *cfg;
  cudaStream_t s = (cudaStream_t)stream;
  if (c.T == 0)
    return cuda_status(launch_router_backward(c, nullptr, nullptr, nullptr, nullptr, 0.0f, nullptr, nullptr, dw_router,
                                              d_router_bias, RouterScratch{}, nullptr, s));
  if (!ptr_ok(logits) || !ptr_ok(topk_idx) || !ptr_ok(dtopk_w) || !ptr_ok(dlogits) || !ptr_ok(ws) ||
      (dw_router && !ptr_ok(x)))
    return MOE_ERR_INVALID_ARG;
  const RouterBwdLayout L = router_bwd_layout(c);
  const RouterScratch sc = router_scratch((char*)ws, L.rpart, L.rbpart, L.dlb, L.dxr, L.roff);
  return cuda_status(launch_router_backward(c, logits, topk_idx, dtopk_w, counts, aux_alpha, x, dlogits, dw_router,
                                            d_router_bias, sc, status_of(ws), s));
}

moe_status_t moe_dispatch_router_backward(const moe_config_t* cfg, const void* dxd, const int32_t* tok_row,
                                          const float* dlogits, const void* w_router, void* dx, void* ws,
                                          moe_stream_t stream) {
  moe_status_t v = validate(cfg);
  if (v != MOE_OK) return v;
  if (cfg->act_dtype != MOE_DTYPE_BF16 || cfg->H % 8) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!ptr_ok(dlogits) || !ptr_ok(w_router) || !ptr_ok(dx) || !ptr_ok(ws) || (dxd && !ptr_ok(tok_row)) ||
      !opt_ok(dxd))
    return MOE_ERR_INVALID_ARG;
  const RouterBwdLayout L = router_bwd_layout(*cfg);
  const RouterScratch sc = router_scratch((char*)ws, L.rpart, L.rbpart, L.dlb, L.dxr, L.roff);
  return cuda_status(launch_router_input_grad(*cfg, dlogits, nullptr, w_router, dxd, tok_row, dx, sc, status_of(ws),
                                              (cudaStream_t)stream));
}

moe_status_t moe_quantize_mx(const void* src_bf16, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                             moe_stream_t stream) {
  if (!ptr_ok(src_bf16) || !ptr_ok(q) || !ptr_ok(sf) || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if (rows % 128 || cols % 128) return MOE_ERR_UNSUPPORTED;
  if (rows * (cols / 32) / 256 >= (int64_t)INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_quantize_mx(src_bf16, rows, cols, q, sf, (cudaStream_t)stream));
}

moe_status_t moe_read_status(void* ws, moe_stream_t stream, int32_t* device_status) {
  if (!ptr_ok(ws) || !device_status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus h{};
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(h), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *device_status = h.code;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_BAD_INPUT: return "device: bad input (expert id out of range, repeated id or non-finite score)";
    case MOE_ERR_TIMEOUT: return "device: bounded wait expired";
  }
  return "unknown status";
}

}  // extern "C"
