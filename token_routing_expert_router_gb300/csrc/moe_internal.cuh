// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------------------
// Workspace layout. The head (4 KB) holds the device status word and, from byte 128, the
// single-launch routing's grid barrier (counter and flag on separate 128-byte lines); the
// routing scan's per-block expert counts follow.
// moe_forward's intermediates come after that.
// ---------------------------------------------------------------------------------------
constexpr size_t kWsHead = 4096;
constexpr int kScanChunk = 128;  // tokens per block of the counting pass

struct DeviceStatus {
  int32_t code;    // first error wins (atomicCAS from 0)
  int32_t detail;  // e.g. the offending token
};

__device__ __forceinline__ void set_status(DeviceStatus* st, int32_t code, int32_t detail) {
  if (atomicCAS(&st->code, 0, code) == 0) st->detail = detail;
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t routed_rows(const moe_config_t& c) { return (int64_t)c.T * c.k; }
inline int64_t total_rows(const moe_config_t& c) { return (int64_t)c.T * c.k + (c.n_shared ? c.T : 0); }
inline int scan_blocks(const moe_config_t& c) { return (int)ceil_div(c.T, kScanChunk); }

// ---------------------------------------------------------------------------------------
// Kernel launchers (one translation unit each; all stream-ordered, no host sync).
// ---------------------------------------------------------------------------------------
cudaError_t launch_route_topk(const moe_config_t& c, const float* logits, int32_t* topk_idx,
                              float* topk_w, DeviceStatus* st, cudaStream_t s);
bool router_small_supported(const moe_config_t& c);
cudaError_t launch_router_small(const moe_config_t& c, const void* x, const void* w, const float* bias,
                                float* logits, cudaStream_t s);
// The auxiliary loss in two launches (part: [ceil(T / 128)][E] 64-bit scratch).
cudaError_t launch_aux_loss(const moe_config_t& c, const float* logits, const int32_t* counts, float alpha,
                            float* loss, uint64_t* part, cudaStream_t s);
// S1 + S2 in one cooperative launch (at most kFusedMaxRouteBlocks blocks): blockcnt holds
// [blocks][E] counts, barrier two words of the workspace head (zero when initialised).
// With auxp ([blocks][E] 64-bit scratch) the same launch writes the auxiliary loss (the value
// launch_aux_loss gives) to *aux_loss.
constexpr int kFusedMaxRouteBlocks = 512;
bool route_fused_supported(const moe_config_t& c);
cudaError_t launch_route_fused(const moe_config_t& c, const float* logits, int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* tok_row,
                               int32_t* blockcnt, uint32_t* barrier, DeviceStatus* st, cudaStream_t s,
                               uint64_t* auxp = nullptr, float aux_alpha = 0.0f, float* aux_loss = nullptr);
cudaError_t launch_route_scan(const moe_config_t& c, const int32_t* topk_idx, int32_t* counts,
                              int32_t* offsets, int32_t* row_token, int32_t* tok_row,
                              int32_t* blockcnt, DeviceStatus* st, cudaStream_t s);
cudaError_t launch_dispatch(const moe_config_t& c, const void* x, const int32_t* tok_row,
                            void* xd, float* xd_scale, cudaStream_t s);
cudaError_t launch_combine(const moe_config_t& c, const void* yd, const int32_t* tok_row,
                           const float* topk_w, void* y, cudaStream_t s);
cudaError_t launch_quantize_e4m3(const void* src, int64_t rows, int64_t cols, int br, int bc,
                                 uint8_t* q, float* scale, cudaStream_t s);
// Backward of combine (bf16 layers): dyd = w * dy (+ shared rows = dy), dtopk_w = <dy, yd>.
// Dispatch backward is launch_combine with topk_w = nullptr (unit weights).
cudaError_t launch_combine_backward(const moe_config_t& c, const void* dy, const void* yd, const int32_t* tok_row,
                                    const float* topk_w, void* dyd, float* dtopk_w, cudaStream_t s);
// MXFP8 variant (scale atoms as described in mx_common.cuh).
cudaError_t launch_dispatch_mx(const moe_config_t& c, const void* x, const int32_t* topk_idx,
                               const int32_t* tok_row, const int32_t* offsets, void* xd, void* xd_sf,
                               cudaStream_t s);
cudaError_t launch_quantize_mx(const void* src, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf,
                               cudaStream_t s);

// Router backward (router_bwd.cu). dl: dL/dlogits [T, E] fp32.
int router_wgrad_slices(const moe_config_t& c);  // token slices of the split reductions
int router_bias_slices(const moe_config_t& c);   // slices of the tensor-core path's bias sum
// token slices of the tensor-core weight gradient: (tokens per slice, slices <= 255)
void router_tc_slices(const moe_config_t& c, int* slice, int* slices);
// true: the two router products run on the tensor cores (dl rounded to bf16)
bool router_backward_tc(const moe_config_t& c);
// Workspace buffers of the router backward: part [S, E, H] fp32 (S = router_wgrad_slices,
// or on the tensor-core path the slices of router_tc_slices), bias_part
// [max(S, router_bias_slices), E] fp32, and on the tensor-core path dl_bf16 [T, E], dx_r
// [T, H] bf16 and slice_offsets [slices + 1].
struct RouterScratch {
  float* part;
  float* bias_part;
  void* dl_bf16;
  void* dx_r;
  int32_t* slice_offsets;
};
// dl from dtopk_w (+ the aux loss's gradient when counts != NULL); with dw_router, the
// router weight gradient and (d_bias != NULL) the bias gradient.
cudaError_t launch_router_backward(const moe_config_t& c, const float* logits, const int32_t* topk_idx,
                                   const float* dtopk_w, const int32_t* counts, float aux_alpha, const void* x,
                                   float* dl, float* dw_router, float* d_bias, const RouterScratch& sc,
                                   DeviceStatus* st, cudaStream_t s);
// dx = dl W_router (+ the dispatch backward's rows when dxd != NULL). dl_bf16: dl already
// in bf16 (from launch_router_backward on the tensor-core path), or NULL.
cudaError_t launch_router_input_grad(const moe_config_t& c, const float* dl, const void* dl_bf16,
                                     const void* w_router, const void* dxd, const int32_t* tok_row, void* dx,
                                     const RouterScratch& sc, DeviceStatus* st, cudaStream_t s);
// The combine kernel with unit weights and one more row, row t of extra [T, H] (bf16).
bool combine_extra_supported(const moe_config_t& c);
cudaError_t launch_combine_extra(const moe_config_t& c, const void* yd, const int32_t* tok_row, const void* extra,
                                 void* y, cudaStream_t s);

// SIMT grouped GEMM (fp32 FFMA): C = A . B^T per group, with optional SwiGLU pair.
// Groups: routed experts g < E over rows [offsets[g], offsets[g+1]) of A, plus an optional
// extra group (shared expert) over rows [0, T) of A2 written at output row R + t.
struct SimtGemmArgs {
  int mode;             // 0: C fp32 (+ bias over columns), 1: SwiGLU -> act, 2: store act
  int act_bf16;         // element type of A, B and the act output: 1 bf16, 0 fp32
  int M_static;         // rows of a single-group problem (router: T); -1 for grouped
  const int32_t* offsets;  // [G+1] device (grouped)
  int G;                // routed groups
  int extra_group;      // 1: shared expert group present
  int64_t routed_rows;  // R = T*k: rows of A covered by the G groups; the extra group's
                        // output rows start at R
  const void* A;        // [rows, K]
  const void* A_extra;  // [T, K] shared-expert A (may equal A + R*K)
  int T_extra;          // rows of the extra group
  const void* B0;       // [G, N, K] (mode 1: gate), or [N, K] single
  const void* B1;       // mode 1: up [G, N, K]
  const void* B0_extra; // shared expert weights [N, K]
  const void* B1_extra;
  const float* bias;    // mode 0: [N] or NULL
  void* C;              // [rows, N]
  int N, K;
};
cudaError_t launch_simt_gemm(const SimtGemmArgs& a, cudaStream_t s);

}  // namespace moe
