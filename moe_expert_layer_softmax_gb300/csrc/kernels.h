// Internal launch interface between the C ABI (api.cu) and the kernel files.
// Every launcher enqueues on `stream` and returns the cudaError_t of the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

// Launch with programmatic stream serialisation (the kernel calls pdl_begin(),
// or pdl_launch_dependents() + pdl_wait(), before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Tokens per routing block: the top-k kernels write one expert histogram per
// block and each route's rank within its expert among the block's routes.
constexpr int kRouteTokensPerBlock = 128;

struct DeviceInfo {
  int sm_count = 0;
  bool ready = false;
};
const DeviceInfo* device_info();

// ---------------------------------------------------------------- routing
cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* gates, int32_t* local_rank, int32_t* block_hist,
                              int32_t* err, cudaStream_t s);
// block_hist [ceil(T / kRouteTokensPerBlock), E] is replaced by each block's
// first row per expert; counts, offsets, tile_offsets written
cudaError_t launch_route_scan(int32_t* block_hist, int n_blocks, int E, int32_t* counts,
                              int32_t* offsets, int32_t* tile_offsets, cudaStream_t s);
cudaError_t launch_route_slots(const int32_t* topk_idx, const int32_t* local_rank,
                               const int32_t* block_base, const int32_t* counts,
                               const int32_t* tile_offsets, int T, int E, int k, int64_t rows_max,
                               int32_t* slot_of_route, int32_t* route_of_slot, int32_t* err,
                               cudaStream_t s);
// The whole routing sequence (moe_route and moe_route_noalloc): the router GEMM
// when w_router is given, a top-k kernel, the scan, the slots.  hist holds
// ceil(T / kRouteTokensPerBlock) * E ints, rank T * k ints.
cudaError_t launch_route(int T, int d, int E, int k, int64_t rows_max, const void* x,
                         const void* w_router, const float* bias, float* logits,
                         int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
                         int32_t* tile_offsets, int32_t* slot_of_route, int32_t* route_of_slot,
                         int32_t* err, int32_t* hist, int32_t* rank, cudaStream_t s);

// ---------------------------------------------------------------- data movement
cudaError_t launch_dispatch_bf16(const void* x, const int32_t* slot_of_route,
                                 const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                                 int E, int k, void* xd, cudaStream_t s);
cudaError_t launch_combine(const void* y, const float* gates, const int32_t* slot_of_route, int T,
                           int d, int E, int k, void* out, cudaStream_t s);
cudaError_t launch_combine_bwd(const void* d_out, const void* y, const float* gates,
                               const int32_t* topk_idx, const int32_t* slot_of_route,
                               const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                               int E, int k, void* dy, float* d_gates, float* dlogits,
                               cudaStream_t s,
                               const float* lb_logits = nullptr, float lb_scale = 0.0f,
                               uint8_t* dyq = nullptr, uint8_t* dys = nullptr);
cudaError_t launch_dispatch_bwd(const void* dxd, const int32_t* slot_of_route,
                                const int32_t* topk_idx, const float* dlogits,
                                const void* w_router, int T, int d, int E, int k, void* dx,
                                cudaStream_t s);
// ---------------------------------------------------------------- load balancing
// LBL = E * sum_e f_e P_e; lb_stats = [LBL, P_0 .. P_{E-1}]; `partial` holds
// lb_partial_blocks(T) * E floats.
int lb_partial_blocks(int T);
cudaError_t launch_load_balance(const float* logits, const int32_t* counts, int T, int E, int k,
                                float* partial, float* lb_stats, cudaStream_t s);
// Dense router backward (every logit may carry gradient): dx = sum_j dXd[slot]
// + dlogits . W_r, and dW_r = dlogits^T . x over router_dense_splits(E) token
// splits (`partial` holds kRouterDenseRows * d floats: splits * E <= 1024).
constexpr int kRouterDenseRows = 1024;
inline int router_dense_splits(int E) {
  const int s = kRouterDenseRows / E;
  return s < 1 ? 1 : (s > 32 ? 32 : s);
}
cudaError_t launch_dispatch_bwd_dense(const void* dxd, const int32_t* slot_of_route,
                                      const float* dlogits, const void* w_router, int T, int d,
                                      int E, int k, void* dx, cudaStream_t s);
cudaError_t launch_router_bwd_dense(const void* x, const float* dlogits, int T, int d, int E,
                                    float* partial, float* dw_router, cudaStream_t s);
cudaError_t launch_router_bwd(const void* x, const float* dlogits, const int32_t* route_of_slot,
                              const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                              int E, int k, int64_t tiles_max, float* partial, float* dw_router,
                              cudaStream_t s);

// ---------------------------------------------------------------- grouped GEMM
enum GemmOp {
  OP_FWD1_SWIGLU = 0,
  OP_FWD2 = 1,
  OP_DGRAD2_SWIGLU = 2,
  OP_DGRAD1 = 3,
  OP_WGRAD2 = 4,
  OP_WGRAD1 = 5,
  OP_ROUTER = 6,
  // MXFP8 (E4M3 operands with E8M0 block scales), K-major operands only
  OP_MX_FWD1_SWIGLU = 7,   // A = Xd_q; B = [W_gate|W_up] cache, 64-row groups alternating
  OP_MX_FWD2 = 8,          // A = A_q;  B = W_down cache
  OP_MX_DGRAD2_SWIGLU = 9, // A = dY_q; B = W_down^T cache
  OP_MX_DGRAD1 = 10,       // A0/A1 = dH_q/dU_q; B0/B1 = W_gate^T / W_up^T caches
  // weight gradients whose activation operand (B) is MXFP8 codes in the
  // forward's row layout, dequantised inside the kernel (scales in sfb0)
  OP_WGRAD2_NAT = 11,      // as OP_WGRAD2 with a1 = A_q
  OP_WGRAD1_NAT = 12,      // as OP_WGRAD1 with aux0 = Xd_q
};
// The in-kernel dequantisation needs 256-column B tiles on CTA pairs: both
// weight-gradient shapes' column counts (N) and WGRAD2's M a multiple of 256.
inline bool natural_wgrad_supported(int op, int d, int f) {
  if (op == OP_WGRAD2_NAT) return d % 256 == 0 && f % 256 == 0;
  if (op == OP_WGRAD1_NAT) return d % 256 == 0;
  return false;
}

struct GemmLaunch {
  int op;
  int T, d, E, f;
  int64_t rows_max;
  const int32_t* tile_offsets;
  const void* a0;
  const void* a1;
  const void* w0;
  const void* w1;
  const void* aux0;
  const void* aux1;
  const float* bias;
  void* out0;
  void* out1;
  void* out2;
  void* out3;
  // MXFP8: operand scales (sf_offset layout) and scales of quantised outputs
  const uint8_t* sfa0;
  const uint8_t* sfa1;
  const uint8_t* sfb0;
  const uint8_t* sfb1;
  uint8_t* osf0;
  uint8_t* osf1;
  int32_t* err;
};
cudaError_t launch_grouped_gemm(const GemmLaunch& g, cudaStream_t s);
// ---------------------------------------------------------------- MXFP8
// block_axis 1 with group > 0 interleaves: output row (r/group)*2*group + offset + r%group
cudaError_t launch_quantize_mxfp8(int batch, int rows, int cols, int block_axis, const void* src,
                                  uint8_t* q, uint8_t* sf, cudaStream_t s, int group = 0,
                                  int offset = 0);
// Both orientations of [batch][rows, cols] bf16 in one pass: blocked along cols
// (row interleave as above) and the transpose [cols, rows] blocked along rows.
cudaError_t launch_quantize_mxfp8_both(int batch, int rows, int cols, const void* src, int group,
                                       int offset, uint8_t* q_rows, uint8_t* sf_rows,
                                       uint8_t* q_cols, uint8_t* sf_cols, cudaStream_t s);
cudaError_t launch_dispatch_mxfp8(const void* x, const int32_t* slot_of_route,
                                  const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                                  int E, int k, uint8_t* xq, uint8_t* xs, cudaStream_t s,
                                  void* xdq = nullptr);
cudaError_t launch_dequantize_mxfp8(const uint8_t* q, const uint8_t* sf, int64_t rows, int K,
                                    void* out, cudaStream_t s);
cudaError_t gemm_init_attributes();
// Check words of the checks build (device addresses; NULL in the normal build),
// one per translation unit with device-data-dependent indexing.
int32_t* check_word_move();
int32_t* check_word_quant();
int32_t* check_word_balance();
int32_t* check_word_gemm();
int32_t* check_word_route();
void noalloc_forget_device(int dev);   // moe_route_noalloc's cached scratch address
int gemm_set_inject_stall(int mode);   // returns the previous mode

}  // namespace moe
