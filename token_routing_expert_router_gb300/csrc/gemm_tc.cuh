// Tensor-core (tcgen05 / TMEM / TMA) paths of the router logits and the grouped expert MLP.
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace tc {

// Shapes the tcgen05 kernels take (bf16 activations; E4M3 / MXE4M3 transfer when configured).
bool router_supported(const moe_config_t& c);
bool mlp_supported(const moe_config_t& c);

cudaError_t launch_router(const moe_config_t& c, const void* x, const void* w_router,
                          const float* bias, float* logits, DeviceStatus* st, cudaStream_t s);

// row_token non-null (bf16 only): GEMM1 gathers its routed A rows from x by token instead
// of reading dispatched rows from xd (xd unused). topk_w non-null (with row_token and
// tok_row): GEMM2 scales each routed row of yd by its routing weight before rounding.
// gu_keep non-null (bf16, not with row_token): GEMM1 also stores g and u [rows, 2F] in the
// layout the backward reads (the recomputed gate/up pre-activations, bit for bit).
cudaError_t launch_grouped_mlp(const moe_config_t& c, const void* xd, const float* xd_scale,
                               const void* x, const int32_t* offsets, const moe_weights_t& w,
                               void* h, float* h_scale, void* yd, DeviceStatus* st,
                               cudaStream_t s, const int32_t* row_token = nullptr,
                               const int32_t* tok_row = nullptr, const float* topk_w = nullptr,
                               void* gu_keep = nullptr);

// The bf16 grouped MLP with the tokens on the MMA's N axis (CTA pairs of 256 weight rows,
// token tiles in multiples of 32): the form for experts with few rows each.
bool swap_supported(const moe_config_t& c);
cudaError_t launch_grouped_mlp_swap(const moe_config_t& c, const void* xd, const void* x, const int32_t* offsets,
                                    const moe_weights_t& w, void* h, void* yd, DeviceStatus* st, cudaStream_t s);

// Backward of the grouped expert MLP (bf16). gu [R(+T), 2F] (g and u in 128-column blocks,
// as the gate/up GEMM's tiles hold them); dgu the same columns and h [., F] with each
// expert's rows padded to a multiple of 64 (backward_padded_rows rows): workspace.
// launch_gate_up_preact is the forward's gate/up GEMM storing g and u (no activation).
bool mlp_backward_supported(const moe_config_t& c);
// Rows of the padded dgu and h buffers (every expert's rows padded to a multiple of 64).
int64_t backward_padded_rows(const moe_config_t& c);
cudaError_t launch_gate_up_preact(const moe_config_t& c, const void* xd, const void* x, const int32_t* offsets,
                                  const moe_weights_t& w, void* gu, DeviceStatus* st, cudaStream_t s);
// gu_ready: gu already holds g and u (kept by the forward), so the gate/up GEMM is not rerun.
cudaError_t launch_grouped_mlp_backward(const moe_config_t& c, const void* xd, const void* x,
                                        const int32_t* offsets, const moe_weights_t& w, const void* dyd, void* gu,
                                        void* dgu, void* h, void* dxd, const moe_weight_grads_t& gr,
                                        DeviceStatus* st, cudaStream_t s, bool gu_ready = false);

// The router's two products for its backward on the tensor cores (bf16, E a multiple of
// 128, H of 256): dw_router = dl^T x (fp32, NULL to skip) and dx_r = dl W_router (bf16 [T, H], NULL
// to skip), dl_bf16 [T, E] the logit gradient rounded to bf16. slices > 1: the weight
// gradient is split over token slices (slice_offsets [slices + 1] on the device, every slice
// but the last a multiple of 64 tokens) and dw_router receives the partial sums [slices, E, H].
bool router_backward_tc_supported(const moe_config_t& c);
cudaError_t launch_router_products(const moe_config_t& c, const void* dl_bf16, const void* x, const void* w_router,
                                   float* dw_router, void* dx_r, DeviceStatus* st, cudaStream_t s,
                                   const int32_t* slice_offsets = nullptr, int slices = 1);

// MXFP8 (e4m3, UE8M0 scale atoms) variant on the block-scaled MMA.
bool mx_supported(const moe_config_t& c);
cudaError_t launch_grouped_mlp_mx(const moe_config_t& c, const void* xd, const void* xd_sf,
                                  const int32_t* offsets, const moe_weights_t& w, void* h, void* h_sf,
                                  void* yd, DeviceStatus* st, cudaStream_t s);

// FP8 (e4m3, fp32 block scales) variant of the grouped MLP.
bool fp8_supported(const moe_config_t& c);
cudaError_t launch_grouped_mlp_fp8(const moe_config_t& c, const void* xd, const float* xd_scale,
                                   const int32_t* offsets, const moe_weights_t& w, void* h,
                                   float* h_scale, void* yd, DeviceStatus* st, cudaStream_t s);

}  // namespace tc
}  // namespace moe
