/*
 * moe.h - C ABI of the GB300 (sm_103a) MoE expert layer library (libmoe_gb300.so).
 *
 * One GPU, one stream, no host synchronisation anywhere on the path.  The layer:
 *
 *   route     router projection (x . W_r^T + bias, fp32), softmax over the experts,
 *             top-k by logit (equal logits: lower expert id first), gates = the
 *             selected probabilities renormalised to sum to one;
 *   counts    per-expert route counts, their exclusive scan and the tile-aligned
 *             expert buffer offsets, all kept on the device;
 *   dispatch  each token row is written straight into its expert's contiguous
 *             buffer (no separate permutation pass);
 *   experts   device-scheduled grouped SwiGLU GEMMs (tcgen05 tensor cores, TMA)
 *             whose tile schedule is read from the device-resident offsets;
 *   combine   out[t] = sum_j gate[t, j] * y[slot(t, j)];
 *   backward  combine / SwiGLU / dispatch / router gradients, data-gradient and
 *             weight-gradient grouped GEMMs.
 *
 * Sources: "Supercharging Olmo-core for Efficient and Scalable MoE Training",
 * Abstract (rowwise dispatch writing each token directly into its expert's
 * buffer, routing metadata kept on the GPU, device-scheduled grouped GEMMs,
 * MXFP8); Section 24 (Conclusion), Evidence 3 / Figure 74 and Section 24.1 (the
 * original path copied the route counts to the host once per routed block; the
 * device-resident metadata removes that wait without changing the routing
 * calculation); Section 24.3 / Evidence 10 (MXFP8 payload of 33/32 byte per
 * value, two weight caches, a quantiser must emit a layout the GEMM consumes
 * without conversion); the blog "Olmo-core 3: an open training stack for
 * trillion-parameter MoE", section "Olmo-core 3's answer: experts resident,
 * data routed" (grouped GEMM over uneven per-expert shapes without padding to a
 * common capacity); Section 24.2 / Evidence 9 (the Switch-style load-balancing
 * scalar) and Section 24.3 / Evidence 11 (per-layer recompute).  The pages do
 * not write the layer's arithmetic out; the readings taken (softmax/top-k/
 * renormalisation, bias-free SwiGLU experts, gate applied in the combine) are
 * listed with each call.
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *     The library never allocates or frees device memory on these paths and
 *     keeps no state between calls except what moe_init() caches per device
 *     (and the CUDA events of the timing hook, created on its first use).
 *   - bf16 tensors are raw 16-bit patterns; all matrices are row-major and
 *     contiguous.  Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void*; all work is enqueued on it and
 *     no call waits for the GPU (except moe_read_error and moe_profile_stop).
 *     moe_layer_fwd / moe_layer_bwd (and the stage calls they are built from)
 *     can be captured into a CUDA graph.
 *   - Return value: MOE_OK (0), or a negative MOE_ERR_* code from host-side
 *     argument validation (nothing is enqueued then) or from a failed launch.
 *   - Conditions found on the device (a non-finite logit, a bounded wait that
 *     ran out) set bits of the 32-bit error word at the start of the workspace
 *     `ws`; read it with moe_read_error().  Outputs stay defined (finite
 *     routing with zero gates for the affected tokens).
 *
 * Shape envelope: 1 <= top_k <= n_experts <= 256; d_model and d_ff multiples
 * of 128; T >= 1; T * top_k < 2^31.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define MOE_OK 0
#define MOE_ERR_INVALID (-1)     /* null pointer, bad size, bad enum value        */
#define MOE_ERR_UNSUPPORTED (-2) /* shape outside the envelope above              */
#define MOE_ERR_ALIGN (-3)       /* a device pointer is not 16-byte aligned       */
#define MOE_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed          */
#define MOE_ERR_NOT_INIT (-5)    /* moe_init() was not called for this device     */
#define MOE_ERR_SCRATCH_LIMIT (-6) /* shape needs more than moe_route_noalloc's fixed scratch */

/* bits of the device error word (first int32 of the workspace) */
#define MOE_DEVERR_NONFINITE_LOGIT 0x1 /* a router logit was NaN/Inf             */
#define MOE_DEVERR_TIMEOUT 0x2         /* a bounded on-chip wait gave up         */
#define MOE_DEVERR_BOUNDS 0x4          /* an index left its buffer (not expected) */

/* rows of one grouped-GEMM tile; every expert buffer is padded to a multiple */
#define MOE_TILE_M 128

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1 } moe_prec_t;

typedef struct {
  int32_t T;         /* tokens                                   */
  int32_t d_model;   /* d                                        */
  int32_t n_experts; /* E                                        */
  int32_t top_k;     /* k                                        */
  int32_t d_ff;      /* f (hidden width of one SwiGLU expert)    */
  int32_t prec;      /* moe_prec_t of the expert GEMMs           */
} moe_shape_t;

/* ---------------------------------------------------------------- set-up */

/* Cache device properties and raise the kernels' shared-memory limits on
 * `device`.  Call once per device (not on the hot path) before the other
 * calls, with that device current. */
MOE_API int moe_init(int device);

/* Upper bound on the rows of the dispatched (expert-contiguous, tile-padded)
 * buffers: T*k + E*(MOE_TILE_M-1), rounded up to MOE_TILE_M.  Pure host
 * arithmetic. */
MOE_API int moe_rows_max(const moe_shape_t* shape, int64_t* rows_max);

/* Bytes of scratch workspace `ws` that the calls below need (error word,
 * per-block histograms, per-route ranks, router-gradient and load-balancing
 * partial sums).  Pure host arithmetic. */
MOE_API int moe_workspace_size(const moe_shape_t* shape, size_t* ws_bytes);

/* Zero the device error word in `ws` (enqueued on `stream`). */
MOE_API int moe_clear_error(void* ws, void* stream);

/* Test hook for the failure path (host-side fault injection; no GPU fault is
 * ever raised).  While `mode` is 1, the TMA producer of every following
 * grouped-GEMM launch issues no copies, so the MMA issuer's bounded wait runs
 * out after about one second: the kernel sets MOE_DEVERR_TIMEOUT in the error
 * word, frees its tensor memory and returns (that launch's outputs are
 * undefined).  mode 0 restores normal operation.  Returns the previous mode. */
MOE_API int moe_debug_inject_stall(int32_t mode);

/* Kernel timing hook (the pages have no counterpart: it serves the benchmark's
 * roofline figure).  moe_profile_start(op) makes every following grouped-GEMM
 * launch of `op` (a moe_gemm_op_t, through moe_grouped_gemm or the layer
 * calls) record a pair of CUDA events around itself on its stream, for up to
 * 1024 launches; the events are created by the library on the first call.
 * moe_profile_stop() waits for those events, writes the summed milliseconds
 * and the number of timed launches, and ends the timing.  Host-side only: no
 * kernel changes.  Not thread-safe against concurrent layer calls. */
MOE_API int moe_profile_start(int32_t op);
MOE_API int moe_profile_stop(float* total_ms, int32_t* launches);

/* Synchronise `stream`, then copy the error word to *code.  Diagnostics only:
 * with moe_profile_stop and moe_checks_read, the only calls that wait for the
 * GPU. */
MOE_API int moe_read_error(const void* ws, int32_t* code, void* stream);

/* Check words of the checks build (the pages have no counterpart: this is test
 * infrastructure standing in for a memory checker).  A library compiled with
 * -DMOE_CHECKS checks every index that a kernel reads from device data (a
 * slot, a route, a padding row, a grouped-GEMM tile's rows) against its buffer
 * before the access: an index outside sets MOE_DEVERR_BOUNDS in a device-side
 * word and the access is skipped.  This call synchronises the device, ORs
 * those words into *flags and clears them when `reset` is not 0.  The normal
 * build has no such words: it returns MOE_ERR_UNSUPPORTED with *flags = 0. */
MOE_API int moe_checks_read(int32_t* flags, int32_t reset);

/* ------------------------------------------------------------ routing (a1-a3)
 * Router projection, softmax/top-k/gates, counts, offsets and stable slots.
 *
 *   x          bf16 [T, d]
 *   w_router   bf16 [E, d], or NULL: then `logits` is an INPUT holding the fp32
 *              router logits [T, E] and the projection is skipped
 *   logit_bias fp32 [T, E] or NULL; added to x . W_r^T
 *   logits     fp32 [T, E]; output (or input, see w_router)
 *   topk_idx   int32 [T, k]  expert of choice j of token t, j-th largest logit
 *   gates      fp32 [T, k]   exp(l_j - l_1) / sum_i exp(l_i - l_1) over the k
 *                            selected logits (= softmax over all E experts,
 *                            renormalised over the selected ones)
 *   counts     int32 [E]     routes per expert
 *   offsets    int32 [E+1]   exclusive scan of counts (offsets[E] = T*k)
 *   tile_offsets int32 [E+1] exclusive scan of ceil(counts/MOE_TILE_M); expert e
 *                            owns rows [128*tile_offsets[e], 128*tile_offsets[e+1])
 *                            of the dispatched buffers (its counts[e] routes
 *                            first, then zero padding)
 *   slot_of_route int32 [T*k] row of route r = t*k + j in the dispatched buffers;
 *                            within an expert, rows follow ascending r
 *   route_of_slot int32 [rows_max] inverse map; -1 on padding rows (entries at
 *                            or past row 128*tile_offsets[E] are left untouched)
 *   ws         workspace of moe_workspace_size() bytes
 *
 * Index outputs are deterministic and independent of the launch configuration.
 */
MOE_API int moe_route(const moe_shape_t* shape, const void* x, const void* w_router,
              const float* logit_bias, float* logits, int32_t* topk_idx, float* gates,
              int32_t* counts, int32_t* offsets, int32_t* tile_offsets,
              int32_t* slot_of_route, int32_t* route_of_slot, void* ws, void* stream);

/* Allocation-free variant of moe_route.  The pages have no counterpart to this
 * call: it exists for callers that cannot hand the library a workspace buffer
 * (plugins hosted by a framework that owns all device memory and exposes no
 * allocator to them; hosts working inside a fixed, pre-assigned memory budget;
 * latency-critical loops that must stay out of cudaMalloc because it can
 * synchronise the whole device and stall work on other streams).
 *
 * Same arguments and results as moe_route, without `ws`.  Its scratch (error
 * word, per-block histograms, per-route ranks) lives in one static device
 * array of 2 MiB inside the library, kept by every GPU that loads the library
 * until the process exits.  Shapes needing more scratch than that
 * (256 + roundup256(ceil(T/128)*E*4) + roundup256(T*k*4) bytes) return
 * MOE_ERR_SCRATCH_LIMIT and queue nothing.  Nothing is allocated.
 *   dev_error  device int32 (nullable): receives the call's device error bits.
 * The first call on a device (and the first after each moe_init of it, e.g.
 * following a device reset) looks up the array's address with that device
 * current; make it before any stream capture starts.  All calls share the array
 * (each clears the error word; the rest is rewritten): calls that overlap on the
 * GPU race and must be serialised by the caller. */
MOE_API int moe_route_noalloc(const moe_shape_t* shape, const void* x, const void* w_router,
                              const float* logit_bias, float* logits, int32_t* topk_idx,
                              float* gates, int32_t* counts, int32_t* offsets,
                              int32_t* tile_offsets, int32_t* slot_of_route,
                              int32_t* route_of_slot, int32_t* dev_error, void* stream);

/* ------------------------------------------------------------ dispatch (a4)
 * Rowwise dispatch: xd[slot_of_route[t*k+j]] = x[t]; padding rows of every
 * expert are written as zeros.  BF16 mode: xd is bf16 [rows_max, d];
 * xd_scales and xd_dq must be NULL.  MXFP8 mode: x[t] is quantised once (a15)
 * and the codes go to xd (uint8 E4M3 [rows_max, d]) and the scales to
 * xd_scales (E8M0, MOE_SF layout below); the payload is 33/32 byte per value.
 * xd_dq (MXFP8 mode, nullable): also the dequantised rows, bf16 [rows_max, d],
 * bit for bit what moe_dequantize_mxfp8 gives for xd (for the BF16 weight
 * gradient). */
MOE_API int moe_dispatch(const moe_shape_t* shape, const void* x, const int32_t* slot_of_route,
                 const int32_t* counts, const int32_t* tile_offsets, void* xd,
                 uint8_t* xd_scales, void* xd_dq, void* stream);

/* ------------------------------------------------------------ MXFP8 (a15)
 * Quantise a bf16 matrix src [rows, cols] with one E8M0 scale per 32
 * consecutive values of the contraction (K) axis.
 *   block_axis = 1: K = cols.  q is uint8 [rows, cols], same orientation.
 *   block_axis = 0: K = rows.  q is the transpose, uint8 [cols, rows] (K-major,
 *                   the orientation the grouped GEMM reads).
 * Scale of a block: 2^s with s the smallest integer such that
 * amax <= 448 * 2^s (s clamped to [-127, 127]; s = 0 for an all-zero block),
 * stored as the byte s + 127.  Codes: E4M3 of value / 2^s, round to nearest
 * even, saturating at +-448.  Rows of the K-major output and its K extent must
 * be multiples of 128.  Scales use the MOE_SF layout:
 *   for a K-major [R, K] operand, the scale of (row r, block b = k/32) is at
 *   byte ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r%128)/32)*4 + (b%4).
 * `batch` matrices of the given shape are processed back to back (src, q and
 * scales advance by one matrix each). */
MOE_API int moe_quantize_mxfp8(int32_t batch, int32_t rows, int32_t cols, int32_t block_axis,
                       const void* src, uint8_t* q, uint8_t* scales, void* stream);

/* Inverse of the quantiser for a K-major MXFP8 operand: out[r][k] =
 * E4M3(q[r][k]) * 2^(scale - 127), stored as bf16 [rows, K] (exact unless the
 * product leaves the bf16 range).  rows and K multiples of 128.  This is the
 * global dequantisation that feeds the BF16 weight-gradient GEMMs ("Supercharging
 * Olmo-core ...", Section 24 Evidence 7 / Table 33). */
MOE_API int moe_dequantize_mxfp8(int64_t rows, int32_t K, const uint8_t* q, const uint8_t* scales,
                                 void* out, void* stream);

/* MXFP8 weight caches, quantised once per weight update ("two weight caches",
 * Section 24 Evidence 10 / Section 24.3): the forward cache is blocked along
 * d_model for W_gate/W_up and along d_ff for W_down; the data-gradient cache
 * holds the transposes, blocked along the other axis.  Every array is K-major
 * for the GEMM that reads it; scales use the MOE_SF layout. */
typedef struct {
  uint8_t* gu_q;    /* [E, 2f, d]  W_gate and W_up rows interleaved in 64-row groups:
                       rows [128j, 128j+64) = W_gate rows [64j, 64j+64),
                       rows [128j+64, 128j+128) = W_up rows [64j, 64j+64)   */
  uint8_t* gu_s;    /* scales of gu_q, E * 2f * d/32 bytes                 */
  uint8_t* down_q;  /* [E, d, f]   W_down, blocks along f                   */
  uint8_t* down_s;
  uint8_t* downT_q; /* [E, f, d]   W_down^T, blocks along d                 */
  uint8_t* downT_s;
  uint8_t* gateT_q; /* [E, d, f]   W_gate^T, blocks along f                 */
  uint8_t* gateT_s;
  uint8_t* upT_q;   /* [E, d, f]   W_up^T, blocks along f                   */
  uint8_t* upT_s;
} moe_mx_weights_t;

/* Fill all MXFP8 weight caches from the bf16 master weights (3 launches: one fused
 * pass per weight writes both of its orientations). */
MOE_API int moe_build_mx_weights(const moe_shape_t* shape, const void* w_gate, const void* w_up,
                                 const void* w_down, const moe_mx_weights_t* cache, void* stream);

/* --------------------------------------------------- grouped GEMMs (a5, a6, a9-a12)
 * Device-scheduled grouped GEMMs on the expert-contiguous buffers.  The tile
 * schedule is read from tile_offsets on the device; no host wait.  Inputs are
 * bf16 with fp32 accumulation in tensor memory (tcgen05); W_gate, W_up are
 * [E, f, d] and W_down [E, d, f].  Row buffers have rows_max rows.
 *
 *   op                    operands (a*, w*, aux*)           outputs (out*)
 *   MOE_GEMM_FWD1_SWIGLU  a0 = Xd [rows,d]; w0 = W_gate,    out0 = H, out1 = U,
 *                         w1 = W_up                         out2 = A = silu(H)*U  (bf16 [rows,f])
 *   MOE_GEMM_FWD2         a0 = A [rows,f]; w0 = W_down      out0 = Y [rows,d] bf16
 *   MOE_GEMM_DGRAD2_SWIGLU a0 = dY [rows,d]; w0 = W_down;   out0 = dH = dA*U*silu'(H),
 *                         aux0 = H, aux1 = U (dA = dY_e W_down_e)  out1 = dU = dA*silu(H)
 *   MOE_GEMM_DGRAD1       a0 = dH, a1 = dU [rows,f];        out0 = dXd = dH W_gate_e + dU W_up_e
 *                         w0 = W_gate, w1 = W_up            (bf16 [rows,d])
 *   MOE_GEMM_WGRAD2       a0 = dY [rows,d], a1 = A [rows,f] out0 = dW_down fp32 [E,d,f]
 *   MOE_GEMM_WGRAD1       a0 = dH, a1 = dU [rows,f],        out0 = dW_gate, out1 = dW_up
 *                         aux0 = Xd [rows,d]                (fp32 [E,f,d])
 * Weight gradients of experts without routes are written as exact zeros.
 */
typedef enum {
  MOE_GEMM_FWD1_SWIGLU = 0,
  MOE_GEMM_FWD2 = 1,
  MOE_GEMM_DGRAD2_SWIGLU = 2,
  MOE_GEMM_DGRAD1 = 3,
  MOE_GEMM_WGRAD2 = 4,
  MOE_GEMM_WGRAD1 = 5,
  MOE_GEMM_WGRAD2_NATURAL = 6,
  MOE_GEMM_WGRAD1_NATURAL = 7
} moe_gemm_op_t;

typedef struct {
  const int32_t* tile_offsets; /* [E+1] from moe_route */
  const void* a0;
  const void* a1;
  const void* w0;
  const void* w1;
  const void* aux0;
  const void* aux1;
  void* out0;
  void* out1;
  void* out2;
  /* MXFP8 only (shape->prec == MOE_MXFP8), see below */
  const uint8_t* sfa0;
  const uint8_t* sfa1;
  const uint8_t* sfb0;
  const uint8_t* sfb1;
  void* out3;
  uint8_t* osf0;
  uint8_t* osf1;
} moe_gemm_args_t;

/* With shape->prec == MOE_MXFP8 the data GEMMs run on tcgen05 block-scaled
 * MXFP8 MMAs (E4M3 x E4M3, E8M0 scales, fp32 accumulation); every a and w operand is
 * uint8 codes with its scales in the matching sf array (MOE_SF layout):
 *   FWD1_SWIGLU   a0 = Xd_q [rows,d]; w0 = gu_q cache      out0 = H, out1 = U (bf16),
 *                                                          out2 = A_q [rows,f], osf0 = its scales,
 *                                                          out3 (nullable) = A dequantised, bf16
 *                                                          [rows,f], bit for bit what
 *                                                          moe_dequantize_mxfp8 gives for A_q
 *   FWD2          a0 = A_q; w0 = down_q cache              out0 = Y (bf16)
 *   DGRAD2_SWIGLU a0 = dY_q [rows,d]; w0 = downT_q cache;  out0 = dH, out1 = dU (bf16),
 *                 aux0 = H, aux1 = U (bf16)                out2 = dH_q, out3 = dU_q, osf0/osf1
 *   DGRAD1        a0 = dH_q, a1 = dU_q; w0 = gateT_q,      out0 = dXd (bf16)
 *                 w1 = upT_q
 * WGRAD1/WGRAD2 stay BF16 (on dequantised activations: the dispatch's xd_dq,
 * FWD1_SWIGLU's out3, or moe_dequantize_mxfp8).
 *
 * Weight gradients on the forward's natural MXFP8 layout ("MXFP8 Wgrad",
 * Section 24.2, Evidence 7 / Table 33 of "Supercharging Olmo-core for
 * Efficient and Scalable MoE Training": a weight-gradient kernel that keeps
 * the row-wise scales instead of converting the operand first).  The
 * activation operand is given as the uint8 E4M3 codes the forward produced
 * (one E8M0 scale per 32 columns of a row, MOE_SF layout, in sfb0) and is
 * dequantised inside the GEMM; the other operand stays bf16.  Either precision
 * mode:
 *   WGRAD2_NATURAL  a0 = dY [rows,d] bf16, a1 = A_q [rows,f], sfb0 = A's scales
 *                   out0 = dW_down fp32 [E,d,f]        (d, f multiples of 256)
 *   WGRAD1_NATURAL  a0 = dH, a1 = dU [rows,f] bf16, aux0 = Xd_q [rows,d],
 *                   sfb0 = Xd's scales; out0 = dW_gate, out1 = dW_up fp32 [E,f,d]
 *                   (d a multiple of 256)
 * The result is bit for bit that of moe_dequantize_mxfp8 followed by
 * WGRAD2/WGRAD1 on the dequantised copy (same bf16 values, same MMA order).
 * Other shapes return MOE_ERR_INVALID. */

MOE_API int moe_grouped_gemm(const moe_shape_t* shape, int32_t op, const moe_gemm_args_t* args,
                     void* ws, void* stream);

/* ------------------------------------------------------------ combine (a7, a8)
 * out[t] = sum_j gates[t,j] * y[slot_of_route[t*k+j]], fp32 sum in j order,
 * stored as bf16 [T, d]. */
MOE_API int moe_combine(const moe_shape_t* shape, const void* y, const float* gates,
                const int32_t* slot_of_route, void* out, void* stream);

/* Combine backward and the first half of the router backward:
 *   d_gates[t,j] = <d_out[t], y[slot(t,j)]>              fp32 [T, k]
 *   dy[slot(t,j)] = gates[t,j] * d_out[t]                 bf16 [rows_max, d]
 *                   (padding rows zeroed)
 *   dlogits[t,e]  = g_j (dg_j - sum_i g_i dg_i) if e = topk_idx[t,j], else 0
 *                   fp32 [T, E] (exact gradient through the renormalised
 *                   softmax for the fixed selection)
 *   dy_q, dy_scales  (both NULL, or both set): the MXFP8 quantisation of dy
 *                   along d (a15) in the same pass, uint8 E4M3 [rows_max, d]
 *                   and E8M0 scales in the MOE_SF layout: byte for byte what
 *                   moe_quantize_mxfp8(block_axis = 1) gives for the bf16 dy
 *                   rows of every tile (padding rows: zero codes, scale 2^0);
 *                   rows past the last tile are not written.  One set without
 *                   the other returns MOE_ERR_INVALID. */
MOE_API int moe_combine_bwd(const moe_shape_t* shape, const void* d_out, const void* y,
                    const float* gates, const int32_t* topk_idx, const int32_t* slot_of_route,
                    const int32_t* counts, const int32_t* tile_offsets, void* dy,
                    float* d_gates, float* dlogits, uint8_t* dy_q, uint8_t* dy_scales,
                    void* stream);

/* ------------------------------------------------- dispatch / router backward (a13, a14)
 * dx[t] = sum_j dxd[slot(t,j)] + sum_j dlogits[t, e_tj] * W_r[e_tj]  (bf16 [T, d];
 * the router term only when w_router != NULL). */
MOE_API int moe_dispatch_bwd(const moe_shape_t* shape, const void* dxd, const int32_t* slot_of_route,
                     const int32_t* topk_idx, const float* dlogits, const void* w_router,
                     void* dx, void* stream);

/* dW_r[e] = sum over routes (t, j) of expert e of dlogits[t, e] * x[t]   (fp32 [E, d]).
 * Deterministic: per-tile partial sums (in `ws`) are added in tile order; an
 * expert without routes gets exact zeros. */
MOE_API int moe_router_bwd(const moe_shape_t* shape, const void* x, const float* dlogits,
                   const int32_t* route_of_slot, const int32_t* counts,
                   const int32_t* tile_offsets, float* dw_router, void* ws, void* stream);

/* ------------------------------------------------------------ load balancing
 * Switch-style load-balancing scalar of the router ("Supercharging Olmo-core
 * for Efficient and Scalable MoE Training", Section 24.2, Evidence 9: a
 * cross-term between soft router scores and hard expert counts):
 *   f_e = counts[e] / (T k)                      hard, not differentiated
 *   P_e = mean over tokens of softmax(logits[t])_e over all E experts
 *   LBL = E * sum_e f_e P_e                      (1 for uniform scores)
 *   lb_stats  fp32 [1 + E]: lb_stats[0] = LBL, lb_stats[1 + e] = P_e.
 * Tokens with a non-finite logit add nothing to P.  Uses `ws` (sized by
 * moe_workspace_size); deterministic (fixed-order sums, no atomics).  The
 * gradient of coef * LBL enters through moe_bwd_args_t.lb_coef. */
MOE_API int moe_load_balance(const moe_shape_t* shape, const float* logits, const int32_t* counts,
                             float* lb_stats, void* ws, void* stream);

/* ------------------------------------------------------------ whole layer
 * Buffers saved by the forward for the backward (all caller-owned, device).
 * Row buffers have rows_max rows (moe_rows_max). */
typedef struct {
  float* logits;          /* [T, E] (input when w_router is NULL)       */
  int32_t* topk_idx;      /* [T, k]                                      */
  float* gates;           /* [T, k]                                      */
  int32_t* counts;        /* [E]                                         */
  int32_t* offsets;       /* [E+1]                                       */
  int32_t* tile_offsets;  /* [E+1]                                       */
  int32_t* slot_of_route; /* [T*k]                                       */
  int32_t* route_of_slot; /* [rows_max]                                  */
  void* xd;               /* bf16 [rows_max, d]                          */
  void* h;                /* bf16 [rows_max, f]                          */
  void* u;                /* bf16 [rows_max, f]                          */
  void* a;                /* bf16 [rows_max, f]                          */
  void* y;                /* bf16 [rows_max, d]                          */
  float* lb_stats;        /* fp32 [1 + E] or NULL: the forward writes the
                             load-balancing statistics here (moe_load_balance) */
} moe_saved_t;

/* MXFP8 activation buffers (rows_max rows; scales in the MOE_SF layout).
 * xd_q/xd_s and a_q/a_s are written by the forward and read by the backward;
 * so are xd_dq and a_dq (the forward writes them when they are non-NULL; the
 * backward needs them, from the forward or from its own recompute); the rest
 * is backward scratch. */
typedef struct moe_mx_buffers {
  uint8_t* xd_q;  /* [rows_max, d] dispatched tokens, quantised once per token */
  uint8_t* xd_s;
  uint8_t* a_q;   /* [rows_max, f] SwiGLU output quantised in the GEMM1 epilogue */
  uint8_t* a_s;
  uint8_t* dy_q;  /* [rows_max, d] */
  uint8_t* dy_s;
  uint8_t* dh_q;  /* [rows_max, f] */
  uint8_t* dh_s;
  uint8_t* du_q;  /* [rows_max, f] */
  uint8_t* du_s;
  void* xd_dq;    /* bf16 [rows_max, d] dequantised Xd for the weight gradients */
  void* a_dq;     /* bf16 [rows_max, f] dequantised A for the weight gradients  */
} moe_mx_buffers_t;

typedef struct {
  const void* x;          /* bf16 [T, d]                                 */
  const void* w_router;   /* bf16 [E, d] or NULL (logits given in saved) */
  const float* logit_bias;/* fp32 [T, E] or NULL                         */
  const void* w_gate;     /* bf16 [E, f, d]                              */
  const void* w_up;       /* bf16 [E, f, d]                              */
  const void* w_down;     /* bf16 [E, d, f]                              */
  void* out;              /* bf16 [T, d]                                 */
  /* MXFP8 only: weight caches and MXFP8 activation buffers (else NULL) */
  const moe_mx_weights_t* mx_weights;
  const struct moe_mx_buffers* mx;
} moe_fwd_args_t;

typedef struct {
  const void* d_out;      /* bf16 [T, d] upstream gradient               */
  const void* x;          /* bf16 [T, d]                                 */
  const void* w_router;   /* bf16 [E, d] or NULL                         */
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  /* outputs */
  void* dx;               /* bf16 [T, d]                                 */
  float* dw_router;       /* fp32 [E, d] (ignored when w_router is NULL) */
  float* dw_gate;         /* fp32 [E, f, d]                              */
  float* dw_up;           /* fp32 [E, f, d]                              */
  float* dw_down;         /* fp32 [E, d, f]                              */
  float* d_gates;         /* fp32 [T, k]                                 */
  float* dlogits;         /* fp32 [T, E]                                 */
  /* gradient buffers (caller-owned scratch, rows_max rows) */
  void* dy;               /* bf16 [rows_max, d]                          */
  void* dh;               /* bf16 [rows_max, f]                          */
  void* du;               /* bf16 [rows_max, f]                          */
  void* dxd;              /* bf16 [rows_max, d]                          */
  /* MXFP8 only (else NULL) */
  const moe_mx_weights_t* mx_weights;
  const moe_mx_buffers_t* mx;
  /* 0: read the expert activations the forward saved.  1: recompute them
   * first (dispatch -> FWD1_SWIGLU -> FWD2 from x and the saved routing
   * metadata), so that saved->xd, h, u, a, y (MXFP8: mx->xd_q/xd_s, a_q/a_s)
   * need not survive from the forward: the caller may reuse that memory in
   * between.  Only x and the routing metadata must be kept. */
  int32_t recompute;
  /* Coefficient of the load-balancing scalar in the loss (0: no such term).
   * When not 0, coef * dLBL/dlogits is added to dlogits for every token and
   * expert, and (with w_router) dx and dW_r take the dense router backward. */
  float lb_coef;
} moe_bwd_args_t;

/* route -> [load-balancing statistics into saved->lb_stats when it is not
 * NULL] -> dispatch -> FWD1_SWIGLU -> FWD2 -> combine, all on `stream`.
 * MXFP8 mode: the dispatch quantises each token once (Xd_q), GEMM1/GEMM2 run
 * on the MXFP8 weight cache, saved->xd and saved->a are not used. */
MOE_API int moe_layer_fwd(const moe_shape_t* shape, const moe_fwd_args_t* args, const moe_saved_t* saved,
                  void* ws, void* stream);

/* [recompute: dispatch -> FWD1_SWIGLU -> FWD2] -> combine_bwd -> DGRAD2_SWIGLU
 * -> WGRAD2 -> DGRAD1 -> WGRAD1 -> dispatch_bwd -> router_bwd, all on `stream`,
 * reading what moe_layer_fwd saved (per-layer recompute: the report's
 * "Section 24: Conclusion", Evidence 11, trades repeated dispatch and expert
 * compute for activation memory).  Recomputed values equal the saved ones bit
 * for bit (the same deterministic kernels on the same inputs).
 * MXFP8 mode: dY is quantised in the combine backward's pass, DGRAD2/DGRAD1 run
 * on MXFP8 (the second weight cache), and the weight gradients run in BF16 on
 * the dequantised Xd and A that the forward (or the recompute) wrote. */
MOE_API int moe_layer_bwd(const moe_shape_t* shape, const moe_bwd_args_t* args, const moe_saved_t* saved,
                  void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
