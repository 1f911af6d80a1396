// C ABI of the MoE expert layer library: argument validation, workspace
// layout, the stage calls and the whole-layer orchestration.  Every call only
// enqueues kernels on the caller's stream; none waits for the GPU except
// moe_read_error.  Declarations and documentation: include/moe.h.
#include <cmath>
#include <cstring>
#include <mutex>

#include "moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const moe_shape_t* s) {
  if (s == nullptr) return MOE_ERR_INVALID;
  if (s->T < 1 || s->d_model < 1 || s->n_experts < 1 || s->top_k < 1 || s->d_ff < 1)
    return MOE_ERR_INVALID;
  if (s->prec != MOE_BF16 && s->prec != MOE_MXFP8) return MOE_ERR_INVALID;
  if (s->top_k > s->n_experts) return MOE_ERR_INVALID;
  if (s->n_experts > 256 || s->top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (s->d_model % 128 != 0 || s->d_ff % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)s->T * s->top_k >= (int64_t(1) << 31) - (int64_t)s->n_experts * kTileM)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int64_t rows_max_of(const moe_shape_t* s) {
  const int64_t R = (int64_t)s->T * s->top_k;
  const int64_t r = R + (int64_t)s->n_experts * (kTileM - 1);
  return (r + kTileM - 1) / kTileM * kTileM;
}

int n_route_blocks(const moe_shape_t* s) {
  return (s->T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
}

// Workspace: [error word | block histograms | route ranks | router-grad partials]
struct WsLayout {
  size_t hist, rank, partial, lb, total;
};
WsLayout ws_layout(const moe_shape_t* s) {
  WsLayout w;
  size_t off = 256;
  w.hist = off;
  off += align256((size_t)n_route_blocks(s) * s->n_experts * 4);
  w.rank = off;
  off += align256((size_t)s->T * s->top_k * 4);
  w.partial = off;   // router-gradient partial sums: per row tile, or per token split (dense)
  const size_t tiles = (size_t)(rows_max_of(s) / kTileM);
  const size_t dense = (size_t)kRouterDenseRows;
  off += align256((tiles > dense ? tiles : dense) * s->d_model * 4);
  w.lb = off;        // load-balancing partial sums
  off += align256((size_t)lb_partial_blocks(s->T) * s->n_experts * 4);
  w.total = off;
  return w;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}

int ready_or_error() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices || !g_dev[dev].ready) return MOE_ERR_NOT_INIT;
  return MOE_OK;
}

#define MOE_TRY(expr)                   \
  do {                                  \
    int _rc = (expr);                   \
    if (_rc != MOE_OK) return _rc;      \
  } while (0)

#define MOE_CUDA(expr)                              \
  do {                                              \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

#define MOE_NONNULL_ALIGNED(p)                   \
  do {                                           \
    if ((p) == nullptr) return MOE_ERR_INVALID;  \
    if (!aligned16(p)) return MOE_ERR_ALIGN;     \
  } while (0)

#define MOE_ALIGNED_OR_NULL(p)                             \
  do {                                                     \
    if ((p) != nullptr && !aligned16(p)) return MOE_ERR_ALIGN; \
  } while (0)

int route_impl(const moe_shape_t* s, const void* x, const void* w_router, const float* bias,
               float* logits, int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
               int32_t* tile_offsets, int32_t* slot_of_route, int32_t* route_of_slot, void* ws,
               cudaStream_t st) {
  const WsLayout w = ws_layout(s);
  int32_t* err = at<int32_t>(ws, 0);
  int32_t* hist = at<int32_t>(ws, w.hist);
  int32_t* rank = at<int32_t>(ws, w.rank);
  MOE_CUDA(launch_route(s->T, s->d_model, s->n_experts, s->top_k, rows_max_of(s), x, w_router, bias,
                        logits, topk_idx, gates, counts, offsets, tile_offsets, slot_of_route,
                        route_of_slot, err, hist, rank, st));
  return MOE_OK;
}

// ---- kernel timing hook (moe_profile_start / moe_profile_stop)
constexpr int kProfMax = 1024;
struct Profile {
  std::mutex mu;
  int op = -1;
  int used = 0;
  cudaEvent_t ev[2 * kProfMax] = {};
  bool created = false;
};
Profile g_prof;

int gemm_impl(const moe_shape_t* s, int op, const moe_gemm_args_t* a, void* ws, cudaStream_t st) {
  GemmLaunch g = {};
  g.op = op;
  if (s->prec == MOE_MXFP8) {
    switch (op) {
      case MOE_GEMM_FWD1_SWIGLU: g.op = OP_MX_FWD1_SWIGLU; break;
      case MOE_GEMM_FWD2: g.op = OP_MX_FWD2; break;
      case MOE_GEMM_DGRAD2_SWIGLU: g.op = OP_MX_DGRAD2_SWIGLU; break;
      case MOE_GEMM_DGRAD1: g.op = OP_MX_DGRAD1; break;
      default: break;   // weight gradients stay BF16
    }
  }
  if (op == MOE_GEMM_WGRAD2_NATURAL) g.op = OP_WGRAD2_NAT;
  if (op == MOE_GEMM_WGRAD1_NATURAL) g.op = OP_WGRAD1_NAT;
  g.sfa0 = a->sfa0; g.sfa1 = a->sfa1; g.sfb0 = a->sfb0; g.sfb1 = a->sfb1;
  g.out3 = a->out3; g.osf0 = a->osf0; g.osf1 = a->osf1;
  g.T = s->T; g.d = s->d_model; g.E = s->n_experts; g.f = s->d_ff;
  g.rows_max = rows_max_of(s);
  g.tile_offsets = a->tile_offsets;
  g.a0 = a->a0; g.a1 = a->a1; g.w0 = a->w0; g.w1 = a->w1;
  g.aux0 = a->aux0; g.aux1 = a->aux1;
  g.out0 = a->out0; g.out1 = a->out1; g.out2 = a->out2;
  g.err = at<int32_t>(ws, 0);
  cudaEvent_t* ev = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.op == op && g_prof.used < kProfMax) ev = &g_prof.ev[2 * g_prof.used++];
  }
  if (ev != nullptr) MOE_CUDA(cudaEventRecord(ev[0], st));
  MOE_CUDA(launch_grouped_gemm(g, st));
  if (ev != nullptr) MOE_CUDA(cudaEventRecord(ev[1], st));
  return MOE_OK;
}

// Operands of the MXFP8 data GEMMs (codes, scales and outputs).
int check_gemm_args_mx(int op, const moe_gemm_args_t* a) {
  if (a == nullptr) return MOE_ERR_INVALID;
  MOE_NONNULL_ALIGNED(a->tile_offsets);
  switch (op) {
    case MOE_GEMM_FWD1_SWIGLU:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->sfa0); MOE_NONNULL_ALIGNED(a->w0);
      MOE_NONNULL_ALIGNED(a->sfb0); MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1);
      MOE_NONNULL_ALIGNED(a->out2); MOE_NONNULL_ALIGNED(a->osf0); MOE_ALIGNED_OR_NULL(a->out3);
      break;
    case MOE_GEMM_FWD2:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->sfa0); MOE_NONNULL_ALIGNED(a->w0);
      MOE_NONNULL_ALIGNED(a->sfb0); MOE_NONNULL_ALIGNED(a->out0);
      break;
    case MOE_GEMM_DGRAD2_SWIGLU:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->sfa0); MOE_NONNULL_ALIGNED(a->w0);
      MOE_NONNULL_ALIGNED(a->sfb0); MOE_NONNULL_ALIGNED(a->aux0); MOE_NONNULL_ALIGNED(a->aux1);
      MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1); MOE_NONNULL_ALIGNED(a->out2);
      MOE_NONNULL_ALIGNED(a->out3); MOE_NONNULL_ALIGNED(a->osf0); MOE_NONNULL_ALIGNED(a->osf1);
      break;
    case MOE_GEMM_DGRAD1:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->sfa0); MOE_NONNULL_ALIGNED(a->a1);
      MOE_NONNULL_ALIGNED(a->sfa1); MOE_NONNULL_ALIGNED(a->w0); MOE_NONNULL_ALIGNED(a->sfb0);
      MOE_NONNULL_ALIGNED(a->w1); MOE_NONNULL_ALIGNED(a->sfb1); MOE_NONNULL_ALIGNED(a->out0);
      break;
    default:
      return MOE_ERR_INVALID;
  }
  return MOE_OK;
}

bool is_mx_data_gemm(int op) {
  return op == MOE_GEMM_FWD1_SWIGLU || op == MOE_GEMM_FWD2 || op == MOE_GEMM_DGRAD2_SWIGLU ||
         op == MOE_GEMM_DGRAD1;
}

int check_mx_buffers(const moe_mx_weights_t* w, const moe_mx_buffers_t* b, bool bwd) {
  if (w == nullptr || b == nullptr) return MOE_ERR_INVALID;
  const void* wp[] = {w->gu_q, w->gu_s, w->down_q, w->down_s, w->downT_q, w->downT_s,
                      w->gateT_q, w->gateT_s, w->upT_q, w->upT_s};
  for (const void* p : wp) MOE_NONNULL_ALIGNED(p);
  MOE_NONNULL_ALIGNED(b->xd_q); MOE_NONNULL_ALIGNED(b->xd_s);
  MOE_NONNULL_ALIGNED(b->a_q); MOE_NONNULL_ALIGNED(b->a_s);
  if (bwd) {
    const void* bp[] = {b->dy_q, b->dy_s, b->dh_q, b->dh_s, b->du_q, b->du_s, b->xd_dq, b->a_dq};
    for (const void* p : bp) MOE_NONNULL_ALIGNED(p);
  }
  return MOE_OK;
}

int check_gemm_args(int op, const moe_gemm_args_t* a) {
  if (a == nullptr) return MOE_ERR_INVALID;
  MOE_NONNULL_ALIGNED(a->tile_offsets);
  switch (op) {
    case MOE_GEMM_FWD1_SWIGLU:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->w0); MOE_NONNULL_ALIGNED(a->w1);
      MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1); MOE_NONNULL_ALIGNED(a->out2);
      break;
    case MOE_GEMM_FWD2:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->w0); MOE_NONNULL_ALIGNED(a->out0);
      break;
    case MOE_GEMM_DGRAD2_SWIGLU:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->w0); MOE_NONNULL_ALIGNED(a->aux0);
      MOE_NONNULL_ALIGNED(a->aux1); MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1);
      break;
    case MOE_GEMM_DGRAD1:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->a1); MOE_NONNULL_ALIGNED(a->w0);
      MOE_NONNULL_ALIGNED(a->w1); MOE_NONNULL_ALIGNED(a->out0);
      break;
    case MOE_GEMM_WGRAD2:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->a1); MOE_NONNULL_ALIGNED(a->out0);
      break;
    case MOE_GEMM_WGRAD1:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->a1); MOE_NONNULL_ALIGNED(a->aux0);
      MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1);
      break;
    case MOE_GEMM_WGRAD2_NATURAL:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->a1); MOE_NONNULL_ALIGNED(a->sfb0);
      MOE_NONNULL_ALIGNED(a->out0);
      break;
    case MOE_GEMM_WGRAD1_NATURAL:
      MOE_NONNULL_ALIGNED(a->a0); MOE_NONNULL_ALIGNED(a->a1); MOE_NONNULL_ALIGNED(a->aux0);
      MOE_NONNULL_ALIGNED(a->sfb0); MOE_NONNULL_ALIGNED(a->out0); MOE_NONNULL_ALIGNED(a->out1);
      break;
    default:
      return MOE_ERR_INVALID;
  }
  return MOE_OK;
}

}  // namespace

const DeviceInfo* device_info() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_dev[dev];
}


// dispatch -> FWD1_SWIGLU -> FWD2: the expert part of the forward, from x and
// the routing metadata in `sv` (writes xd, h, u, a, y; in MXFP8 mode xd_q/xd_s
// and a_q/a_s instead of xd and a).  The backward's recompute mode re-runs it.
int expert_forward(const moe_shape_t* s, const void* x, const void* w_gate, const void* w_up,
                   const void* w_down, const moe_mx_weights_t* w, const moe_mx_buffers_t* b,
                   const moe_saved_t* sv, void* ws, cudaStream_t st) {
  moe_gemm_args_t g = {};
  if (s->prec == MOE_MXFP8) {
    // the dequantised Xd and A (for the weight gradients) come out of the same passes
    MOE_CUDA(launch_dispatch_mxfp8(x, sv->slot_of_route, sv->counts, sv->tile_offsets, s->T,
                                   s->d_model, s->n_experts, s->top_k, b->xd_q, b->xd_s, st,
                                   b->xd_dq));
    g.tile_offsets = sv->tile_offsets;
    g.a0 = b->xd_q; g.sfa0 = b->xd_s; g.w0 = w->gu_q; g.sfb0 = w->gu_s;
    g.out0 = sv->h; g.out1 = sv->u; g.out2 = b->a_q; g.osf0 = b->a_s; g.out3 = b->a_dq;
    MOE_TRY(gemm_impl(s, MOE_GEMM_FWD1_SWIGLU, &g, ws, st));
    g = moe_gemm_args_t{};
    g.tile_offsets = sv->tile_offsets;
    g.a0 = b->a_q; g.sfa0 = b->a_s; g.w0 = w->down_q; g.sfb0 = w->down_s; g.out0 = sv->y;
    return gemm_impl(s, MOE_GEMM_FWD2, &g, ws, st);
  }
  MOE_CUDA(launch_dispatch_bf16(x, sv->slot_of_route, sv->counts, sv->tile_offsets, s->T,
                                s->d_model, s->n_experts, s->top_k, sv->xd, st));
  g.tile_offsets = sv->tile_offsets;
  g.a0 = sv->xd; g.w0 = w_gate; g.w1 = w_up;
  g.out0 = sv->h; g.out1 = sv->u; g.out2 = sv->a;
  MOE_TRY(gemm_impl(s, MOE_GEMM_FWD1_SWIGLU, &g, ws, st));
  g = moe_gemm_args_t{};
  g.tile_offsets = sv->tile_offsets;
  g.a0 = sv->a; g.w0 = w_down; g.out0 = sv->y;
  return gemm_impl(s, MOE_GEMM_FWD2, &g, ws, st);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_init(int device) {
  if (device < 0 || device >= kMaxDevices) return MOE_ERR_INVALID;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != device) return MOE_ERR_INVALID;
  int sms = 0;
  MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  MOE_CUDA(gemm_init_attributes());
  noalloc_forget_device(device);
  g_dev[device].sm_count = sms;
  g_dev[device].ready = true;
  return MOE_OK;
}

int moe_rows_max(const moe_shape_t* shape, int64_t* rows_max) {
  MOE_TRY(check_shape(shape));
  if (rows_max == nullptr) return MOE_ERR_INVALID;
  *rows_max = rows_max_of(shape);
  return MOE_OK;
}

int moe_workspace_size(const moe_shape_t* shape, size_t* ws_bytes) {
  MOE_TRY(check_shape(shape));
  if (ws_bytes == nullptr) return MOE_ERR_INVALID;
  *ws_bytes = ws_layout(shape).total;
  return MOE_OK;
}

int moe_checks_read(int32_t* flags, int32_t reset) {
  if (flags == nullptr) return MOE_ERR_INVALID;
  *flags = 0;
  int32_t* words[] = {check_word_move(), check_word_quant(), check_word_balance(),
                      check_word_gemm(), check_word_route()};
  bool any = false;
  for (int32_t* w : words) {
    if (w == nullptr) continue;
    any = true;
    int32_t v = 0;
    MOE_CUDA(cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost));
    *flags |= v;
    if (reset) MOE_CUDA(cudaMemset(w, 0, sizeof(int32_t)));
  }
  return any ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

int moe_clear_error(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID;
  MOE_CUDA(cudaMemsetAsync(ws, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_debug_inject_stall(int32_t mode) {
  if (mode != 0 && mode != 1) return MOE_ERR_INVALID;
  return gemm_set_inject_stall(mode);
}

int moe_profile_start(int32_t op) {
  if (op < MOE_GEMM_FWD1_SWIGLU || op > MOE_GEMM_WGRAD1) return MOE_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  if (!g_prof.created) {
    for (int i = 0; i < 2 * kProfMax; ++i)
      if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) return MOE_ERR_CUDA;
    g_prof.created = true;
  }
  g_prof.used = 0;
  g_prof.op = op;
  return MOE_OK;
}

int moe_profile_stop(float* total_ms, int32_t* launches) {
  if (total_ms == nullptr || launches == nullptr) return MOE_ERR_INVALID;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.op = -1;
  float sum = 0.0f;
  for (int i = 0; i < g_prof.used; ++i) {
    MOE_CUDA(cudaEventSynchronize(g_prof.ev[2 * i + 1]));
    float ms = 0.0f;
    MOE_CUDA(cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]));
    sum += ms;
  }
  *total_ms = sum;
  *launches = g_prof.used;
  g_prof.used = 0;
  return MOE_OK;
}

int moe_read_error(const void* ws, int32_t* code, void* stream) {
  if (ws == nullptr || code == nullptr) return MOE_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaMemcpyAsync(code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
  MOE_CUDA(cudaStreamSynchronize(st));
  return MOE_OK;
}

int moe_route(const moe_shape_t* s, const void* x, const void* w_router, const float* logit_bias,
              float* logits, int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
              int32_t* tile_offsets, int32_t* slot_of_route, int32_t* route_of_slot, void* ws,
              void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  if (w_router != nullptr) {
    MOE_NONNULL_ALIGNED(x);
    MOE_NONNULL_ALIGNED(w_router);
  }
  MOE_ALIGNED_OR_NULL(logit_bias);
  MOE_NONNULL_ALIGNED(logits);
  MOE_NONNULL_ALIGNED(topk_idx);
  MOE_NONNULL_ALIGNED(gates);
  MOE_NONNULL_ALIGNED(counts);
  MOE_NONNULL_ALIGNED(offsets);
  MOE_NONNULL_ALIGNED(tile_offsets);
  MOE_NONNULL_ALIGNED(slot_of_route);
  MOE_NONNULL_ALIGNED(route_of_slot);
  MOE_NONNULL_ALIGNED(ws);
  return route_impl(s, x, w_router, logit_bias, logits, topk_idx, gates, counts, offsets,
                    tile_offsets, slot_of_route, route_of_slot, ws,
                    static_cast<cudaStream_t>(stream));
}

int moe_dispatch(const moe_shape_t* s, const void* x, const int32_t* slot_of_route,
                 const int32_t* counts, const int32_t* tile_offsets, void* xd, uint8_t* xd_scales,
                 void* xd_dq, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(x);
  MOE_NONNULL_ALIGNED(slot_of_route);
  MOE_NONNULL_ALIGNED(counts);
  MOE_NONNULL_ALIGNED(tile_offsets);
  MOE_NONNULL_ALIGNED(xd);
  if (s->prec == MOE_MXFP8) {
    MOE_NONNULL_ALIGNED(xd_scales);
    MOE_ALIGNED_OR_NULL(xd_dq);
    MOE_CUDA(launch_dispatch_mxfp8(x, slot_of_route, counts, tile_offsets, s->T, s->d_model,
                                   s->n_experts, s->top_k, static_cast<uint8_t*>(xd), xd_scales,
                                   static_cast<cudaStream_t>(stream), xd_dq));
    return MOE_OK;
  }
  if (xd_scales != nullptr || xd_dq != nullptr) return MOE_ERR_INVALID;
  MOE_CUDA(launch_dispatch_bf16(x, slot_of_route, counts, tile_offsets, s->T, s->d_model,
                                s->n_experts, s->top_k, xd, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_quantize_mxfp8(int32_t batch, int32_t rows, int32_t cols, int32_t block_axis,
                       const void* src, uint8_t* q, uint8_t* scales, void* stream) {
  MOE_TRY(ready_or_error());
  if (batch < 1 || rows < 1 || cols < 1 || (block_axis != 0 && block_axis != 1))
    return MOE_ERR_INVALID;
  if (rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NONNULL_ALIGNED(src);
  MOE_NONNULL_ALIGNED(q);
  MOE_NONNULL_ALIGNED(scales);
  MOE_CUDA(launch_quantize_mxfp8(batch, rows, cols, block_axis, src, q, scales,
                                 static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_dequantize_mxfp8(int64_t rows, int32_t K, const uint8_t* q, const uint8_t* scales,
                         void* out, void* stream) {
  MOE_TRY(ready_or_error());
  if (rows < 1 || K < 1) return MOE_ERR_INVALID;
  if (rows % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MOE_NONNULL_ALIGNED(q);
  MOE_NONNULL_ALIGNED(scales);
  MOE_NONNULL_ALIGNED(out);
  MOE_CUDA(launch_dequantize_mxfp8(q, scales, rows, K, out, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_build_mx_weights(const moe_shape_t* s, const void* w_gate, const void* w_up,
                         const void* w_down, const moe_mx_weights_t* c, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  if (c == nullptr) return MOE_ERR_INVALID;
  MOE_NONNULL_ALIGNED(w_gate);
  MOE_NONNULL_ALIGNED(w_up);
  MOE_NONNULL_ALIGNED(w_down);
  const void* ptrs[] = {c->gu_q, c->gu_s, c->down_q, c->down_s, c->downT_q, c->downT_s,
                        c->gateT_q, c->gateT_s, c->upT_q, c->upT_s};
  for (const void* p : ptrs) MOE_NONNULL_ALIGNED(p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = s->n_experts, d = s->d_model, f = s->d_ff;
  // one pass per weight writes both caches: the forward cache (gate/up along d,
  // interleaved in 64-row groups; down along f) and the data-gradient cache
  // (the transposes, blocked along the other axis)
  MOE_CUDA(launch_quantize_mxfp8_both(E, f, d, w_gate, 64, 0, c->gu_q, c->gu_s, c->gateT_q,
                                      c->gateT_s, st));
  MOE_CUDA(launch_quantize_mxfp8_both(E, f, d, w_up, 64, 64, c->gu_q, c->gu_s, c->upT_q,
                                      c->upT_s, st));
  MOE_CUDA(launch_quantize_mxfp8_both(E, d, f, w_down, 0, 0, c->down_q, c->down_s, c->downT_q,
                                      c->downT_s, st));
  return MOE_OK;
}

int moe_grouped_gemm(const moe_shape_t* s, int32_t op, const moe_gemm_args_t* args, void* ws,
                     void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  if (s->prec == MOE_MXFP8 && is_mx_data_gemm(op))
    MOE_TRY(check_gemm_args_mx(op, args));
  else
    MOE_TRY(check_gemm_args(op, args));
  if (op == MOE_GEMM_WGRAD2_NATURAL &&
      !natural_wgrad_supported(OP_WGRAD2_NAT, s->d_model, s->d_ff))
    return MOE_ERR_INVALID;
  if (op == MOE_GEMM_WGRAD1_NATURAL &&
      !natural_wgrad_supported(OP_WGRAD1_NAT, s->d_model, s->d_ff))
    return MOE_ERR_INVALID;
  MOE_NONNULL_ALIGNED(ws);
  return gemm_impl(s, op, args, ws, static_cast<cudaStream_t>(stream));
}

int moe_combine(const moe_shape_t* s, const void* y, const float* gates,
                const int32_t* slot_of_route, void* out, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(y);
  MOE_NONNULL_ALIGNED(gates);
  MOE_NONNULL_ALIGNED(slot_of_route);
  MOE_NONNULL_ALIGNED(out);
  MOE_CUDA(launch_combine(y, gates, slot_of_route, s->T, s->d_model, s->n_experts, s->top_k, out,
                          static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_combine_bwd(const moe_shape_t* s, const void* d_out, const void* y, const float* gates,
                    const int32_t* topk_idx, const int32_t* slot_of_route, const int32_t* counts,
                    const int32_t* tile_offsets, void* dy, float* d_gates, float* dlogits,
                    uint8_t* dy_q, uint8_t* dy_scales, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(d_out);
  MOE_NONNULL_ALIGNED(y);
  MOE_NONNULL_ALIGNED(gates);
  MOE_NONNULL_ALIGNED(topk_idx);
  MOE_NONNULL_ALIGNED(slot_of_route);
  MOE_NONNULL_ALIGNED(counts);
  MOE_NONNULL_ALIGNED(tile_offsets);
  MOE_NONNULL_ALIGNED(dy);
  MOE_NONNULL_ALIGNED(d_gates);
  MOE_ALIGNED_OR_NULL(dlogits);
  MOE_ALIGNED_OR_NULL(dy_q);
  MOE_ALIGNED_OR_NULL(dy_scales);
  if ((dy_q == nullptr) != (dy_scales == nullptr)) return MOE_ERR_INVALID;
  MOE_CUDA(launch_combine_bwd(d_out, y, gates, topk_idx, slot_of_route, counts, tile_offsets, s->T,
                              s->d_model, s->n_experts, s->top_k, dy, d_gates, dlogits,
                              static_cast<cudaStream_t>(stream), nullptr, 0.0f, dy_q, dy_scales));
  return MOE_OK;
}

int moe_dispatch_bwd(const moe_shape_t* s, const void* dxd, const int32_t* slot_of_route,
                     const int32_t* topk_idx, const float* dlogits, const void* w_router,
                     void* dx, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(dxd);
  MOE_NONNULL_ALIGNED(slot_of_route);
  MOE_NONNULL_ALIGNED(topk_idx);
  MOE_NONNULL_ALIGNED(dx);
  MOE_ALIGNED_OR_NULL(w_router);
  if (w_router != nullptr) MOE_NONNULL_ALIGNED(dlogits);
  MOE_CUDA(launch_dispatch_bwd(dxd, slot_of_route, topk_idx, dlogits, w_router, s->T, s->d_model,
                               s->n_experts, s->top_k, dx, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_router_bwd(const moe_shape_t* s, const void* x, const float* dlogits,
                   const int32_t* route_of_slot, const int32_t* counts,
                   const int32_t* tile_offsets, float* dw_router, void* ws, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(x);
  MOE_NONNULL_ALIGNED(dlogits);
  MOE_NONNULL_ALIGNED(route_of_slot);
  MOE_NONNULL_ALIGNED(counts);
  MOE_NONNULL_ALIGNED(tile_offsets);
  MOE_NONNULL_ALIGNED(dw_router);
  MOE_NONNULL_ALIGNED(ws);
  const WsLayout w = ws_layout(s);
  MOE_CUDA(launch_router_bwd(x, dlogits, route_of_slot, counts, tile_offsets, s->T, s->d_model,
                             s->n_experts, s->top_k, rows_max_of(s) / kTileM,
                             at<float>(ws, w.partial), dw_router,
                             static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_load_balance(const moe_shape_t* s, const float* logits, const int32_t* counts,
                     float* lb_stats, void* ws, void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  MOE_NONNULL_ALIGNED(logits);
  MOE_NONNULL_ALIGNED(counts);
  MOE_NONNULL_ALIGNED(lb_stats);
  MOE_NONNULL_ALIGNED(ws);
  const WsLayout w = ws_layout(s);
  MOE_CUDA(launch_load_balance(logits, counts, s->T, s->n_experts, s->top_k, at<float>(ws, w.lb),
                               lb_stats, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_layer_fwd(const moe_shape_t* s, const moe_fwd_args_t* a, const moe_saved_t* sv, void* ws,
                  void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  if (a == nullptr || sv == nullptr) return MOE_ERR_INVALID;
  const bool mx = s->prec == MOE_MXFP8;
  if (mx) MOE_TRY(check_mx_buffers(a->mx_weights, a->mx, false));
  MOE_NONNULL_ALIGNED(a->x);
  MOE_ALIGNED_OR_NULL(a->w_router);
  MOE_ALIGNED_OR_NULL(a->logit_bias);
  MOE_NONNULL_ALIGNED(a->w_gate);
  MOE_NONNULL_ALIGNED(a->w_up);
  MOE_NONNULL_ALIGNED(a->w_down);
  MOE_NONNULL_ALIGNED(a->out);
  MOE_NONNULL_ALIGNED(sv->logits);
  MOE_NONNULL_ALIGNED(sv->topk_idx);
  MOE_NONNULL_ALIGNED(sv->gates);
  MOE_NONNULL_ALIGNED(sv->counts);
  MOE_NONNULL_ALIGNED(sv->offsets);
  MOE_NONNULL_ALIGNED(sv->tile_offsets);
  MOE_NONNULL_ALIGNED(sv->slot_of_route);
  MOE_NONNULL_ALIGNED(sv->route_of_slot);
  if (!mx) {
    MOE_NONNULL_ALIGNED(sv->xd);
    MOE_NONNULL_ALIGNED(sv->a);
  }
  MOE_NONNULL_ALIGNED(sv->h);
  MOE_NONNULL_ALIGNED(sv->u);
  MOE_NONNULL_ALIGNED(sv->y);
  MOE_NONNULL_ALIGNED(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(route_impl(s, a->x, a->w_router, a->logit_bias, sv->logits, sv->topk_idx, sv->gates,
                     sv->counts, sv->offsets, sv->tile_offsets, sv->slot_of_route,
                     sv->route_of_slot, ws, st));
  if (sv->lb_stats != nullptr) {
    MOE_ALIGNED_OR_NULL(sv->lb_stats);
    const WsLayout w = ws_layout(s);
    MOE_CUDA(launch_load_balance(sv->logits, sv->counts, s->T, s->n_experts, s->top_k,
                                 at<float>(ws, w.lb), sv->lb_stats, st));
  }
  MOE_TRY(expert_forward(s, a->x, a->w_gate, a->w_up, a->w_down, a->mx_weights, a->mx, sv, ws, st));
  MOE_CUDA(launch_combine(sv->y, sv->gates, sv->slot_of_route, s->T, s->d_model, s->n_experts, s->top_k, a->out,
                          st));
  return MOE_OK;
}

int moe_layer_bwd(const moe_shape_t* s, const moe_bwd_args_t* a, const moe_saved_t* sv, void* ws,
                  void* stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(ready_or_error());
  if (a == nullptr || sv == nullptr) return MOE_ERR_INVALID;
  const bool mx = s->prec == MOE_MXFP8;
  if (mx) MOE_TRY(check_mx_buffers(a->mx_weights, a->mx, true));
  MOE_NONNULL_ALIGNED(a->d_out);
  MOE_NONNULL_ALIGNED(a->x);
  MOE_ALIGNED_OR_NULL(a->w_router);
  MOE_NONNULL_ALIGNED(a->w_gate);
  MOE_NONNULL_ALIGNED(a->w_up);
  MOE_NONNULL_ALIGNED(a->w_down);
  MOE_NONNULL_ALIGNED(a->dx);
  if (a->w_router != nullptr) MOE_NONNULL_ALIGNED(a->dw_router);
  MOE_NONNULL_ALIGNED(a->dw_gate);
  MOE_NONNULL_ALIGNED(a->dw_up);
  MOE_NONNULL_ALIGNED(a->dw_down);
  MOE_NONNULL_ALIGNED(a->d_gates);
  MOE_NONNULL_ALIGNED(a->dlogits);
  MOE_NONNULL_ALIGNED(a->dy);
  MOE_NONNULL_ALIGNED(a->dh);
  MOE_NONNULL_ALIGNED(a->du);
  MOE_NONNULL_ALIGNED(a->dxd);
  MOE_NONNULL_ALIGNED(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a->recompute != 0 && a->recompute != 1) return MOE_ERR_INVALID;
  if (a->recompute)
    MOE_TRY(expert_forward(s, a->x, a->w_gate, a->w_up, a->w_down, a->mx_weights, a->mx, sv, ws,
                           st));
  // load-balancing term: coef * LBL's gradient joins dlogits (all experts)
  if (!isfinite(a->lb_coef)) return MOE_ERR_INVALID;
  const bool lb = a->lb_coef != 0.0f;
  const float lb_scale = lb ? a->lb_coef * (float)s->n_experts / (float)s->T : 0.0f;
  // MXFP8: dY is quantised along d (for GEMM2's data gradient) in the same pass
  MOE_CUDA(launch_combine_bwd(a->d_out, sv->y, sv->gates, sv->topk_idx, sv->slot_of_route,
                              sv->counts, sv->tile_offsets, s->T, s->d_model, s->n_experts,
                              s->top_k, a->dy, a->d_gates, a->dlogits, st, sv->logits, lb_scale,
                              mx ? a->mx->dy_q : nullptr, mx ? a->mx->dy_s : nullptr));
  if (mx) {
    const moe_mx_weights_t* w = a->mx_weights;
    const moe_mx_buffers_t* b = a->mx;
    moe_gemm_args_t g = {};
    g.tile_offsets = sv->tile_offsets;
    g.a0 = b->dy_q; g.sfa0 = b->dy_s; g.w0 = w->downT_q; g.sfb0 = w->downT_s;
    g.aux0 = sv->h; g.aux1 = sv->u;
    g.out0 = a->dh; g.out1 = a->du; g.out2 = b->dh_q; g.out3 = b->du_q;
    g.osf0 = b->dh_s; g.osf1 = b->du_s;
    MOE_TRY(gemm_impl(s, MOE_GEMM_DGRAD2_SWIGLU, &g, ws, st));
    g = moe_gemm_args_t{};
    g.tile_offsets = sv->tile_offsets;
    g.a0 = a->dy; g.a1 = b->a_dq; g.out0 = a->dw_down;
    MOE_TRY(gemm_impl(s, MOE_GEMM_WGRAD2, &g, ws, st));
    g = moe_gemm_args_t{};
    g.tile_offsets = sv->tile_offsets;
    g.a0 = b->dh_q; g.sfa0 = b->dh_s; g.a1 = b->du_q; g.sfa1 = b->du_s;
    g.w0 = w->gateT_q; g.sfb0 = w->gateT_s; g.w1 = w->upT_q; g.sfb1 = w->upT_s;
    g.out0 = a->dxd;
    MOE_TRY(gemm_impl(s, MOE_GEMM_DGRAD1, &g, ws, st));
    g = moe_gemm_args_t{};
    g.tile_offsets = sv->tile_offsets;
    g.a0 = a->dh; g.a1 = a->du; g.aux0 = b->xd_dq; g.out0 = a->dw_gate; g.out1 = a->dw_up;
    MOE_TRY(gemm_impl(s, MOE_GEMM_WGRAD1, &g, ws, st));
  } else {
  moe_gemm_args_t g = {};
  g.tile_offsets = sv->tile_offsets;
  g.a0 = a->dy; g.w0 = a->w_down; g.aux0 = sv->h; g.aux1 = sv->u;
  g.out0 = a->dh; g.out1 = a->du;
  MOE_TRY(gemm_impl(s, MOE_GEMM_DGRAD2_SWIGLU, &g, ws, st));
  g = moe_gemm_args_t{};
  g.tile_offsets = sv->tile_offsets;
  g.a0 = a->dy; g.a1 = sv->a; g.out0 = a->dw_down;
  MOE_TRY(gemm_impl(s, MOE_GEMM_WGRAD2, &g, ws, st));
  g = moe_gemm_args_t{};
  g.tile_offsets = sv->tile_offsets;
  g.a0 = a->dh; g.a1 = a->du; g.w0 = a->w_gate; g.w1 = a->w_up; g.out0 = a->dxd;
  MOE_TRY(gemm_impl(s, MOE_GEMM_DGRAD1, &g, ws, st));
  g = moe_gemm_args_t{};
  g.tile_offsets = sv->tile_offsets;
  g.a0 = a->dh; g.a1 = a->du; g.aux0 = sv->xd; g.out0 = a->dw_gate; g.out1 = a->dw_up;
  MOE_TRY(gemm_impl(s, MOE_GEMM_WGRAD1, &g, ws, st));
  }
  const WsLayout w = ws_layout(s);
  if (lb && a->w_router != nullptr) {
    // every logit carries gradient: the router backward is dense
    MOE_CUDA(launch_dispatch_bwd_dense(a->dxd, sv->slot_of_route, a->dlogits, a->w_router, s->T,
                                       s->d_model, s->n_experts, s->top_k, a->dx, st));
    MOE_CUDA(launch_router_bwd_dense(a->x, a->dlogits, s->T, s->d_model, s->n_experts,
                                     at<float>(ws, w.partial), a->dw_router, st));
    return MOE_OK;
  }
  MOE_CUDA(launch_dispatch_bwd(a->dxd, sv->slot_of_route, sv->topk_idx, a->dlogits, a->w_router,
                               s->T, s->d_model, s->n_experts, s->top_k, a->dx, st));
  if (a->w_router != nullptr) {
    MOE_CUDA(launch_router_bwd(a->x, a->dlogits, sv->route_of_slot, sv->counts, sv->tile_offsets,
                               s->T, s->d_model, s->n_experts, s->top_k,
                               rows_max_of(s) / kTileM, at<float>(ws, w.partial), a->dw_router,
                               st));
  }
  return MOE_OK;
}

}  // extern "C"
