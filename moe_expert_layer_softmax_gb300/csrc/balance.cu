// Load-balancing statistics and the dense router backward (sm_103a).
//
// "Supercharging Olmo-core for Efficient and Scalable MoE Training", Section
// 24.2 (Evidence 9): the Switch-style load-balancing scalar is a cross-term
// between soft router scores and hard expert counts.  Here
//     f_e = count_e / (T k)            (hard, not differentiated)
//     P_e = mean_t softmax(logits[t])_e (soft, over all E experts)
//     LBL = E * sum_e f_e P_e
// and its gradient, coef * E / T * p[t,e] (f_e - sum_e' f_e' p[t,e']), reaches
// every (token, expert) logit, so with the term on the router backward is
// dense:
//     dx[t]  = sum_j dXd[slot(t, j)] + sum_e dlogits[t, e] W_r[e]
//     dW_r[e] = sum_t dlogits[t, e] x[t]
// All sums run in a fixed order (deterministic, no atomics).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kLbTokensPerBlock = 64;   // 8 warps x 8 tokens

// Per block of 64 tokens: partial[b][e] = sum over the block's tokens of the
// full softmax probability of expert e.  Tokens with a non-finite logit add
// nothing (the routing flags them).
template <int EPL>
__global__ void __launch_bounds__(256) lb_partial_kernel(const float* __restrict__ logits, int T,
                                                         int E, float* __restrict__ partial) {
  pdl_begin();
  __shared__ float s_part[8][256];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.0f;
  const int t0 = blockIdx.x * kLbTokensPerBlock + warp * 8;
  for (int u = 0; u < 8; ++u) {
    const int t = t0 + u;
    if (t >= T) break;   // warp-uniform
    float v[EPL];
    bool bad = false;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? __ldg(logits + (size_t)t * E + e) : -INFINITY;
      if (e < E && !isfinite(v[i])) bad = true;
      mx = fmaxf(mx, v[i]);
    }
    if (__any_sync(0xffffffffu, bad)) continue;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      v[i] = (lane + 32 * i < E) ? expf(v[i] - mx) : 0.0f;
      z += v[i];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv = 1.0f / z;
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] += v[i] * inv;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) s_part[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.0f;
    for (int w = 0; w < 8; ++w) sum += s_part[w][e];
    partial[(size_t)blockIdx.x * E + e] = sum;
  }
}

// lb_stats[0] = LBL, lb_stats[1 + e] = P_e.
__global__ void __launch_bounds__(256) lb_finish_kernel(const float* __restrict__ partial,
                                                        int n_blocks, const int32_t* __restrict__ counts,
                                                        int T, int E, int k, float* __restrict__ lb_stats) {
  pdl_begin();
  __shared__ float s_prod[256];
  const int e = threadIdx.x;
  float prod = 0.0f;
  if (e < E) {
    float sum = 0.0f;
    for (int b = 0; b < n_blocks; ++b) sum += partial[(size_t)b * E + e];
    const float P = sum / (float)T;
    const float f = (float)counts[e] / ((float)T * (float)k);
    lb_stats[1 + e] = P;
    prod = f * P;
  }
  s_prod[threadIdx.x] = prod;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.0f;
    for (int i = 0; i < E; ++i) s += s_prod[i];
    lb_stats[0] = (float)E * s;
  }
}

// ---- dense router backward
constexpr int kDenseTok = 32;    // tokens per block (dx)
constexpr int kDenseCols = 64;   // columns per block: 8 column groups of 8
constexpr int kDenseE = 64;      // experts staged in shared memory at a time

// dx[t] = sum_j dXd[slot(t, j)] + sum_e dlogits[t, e] W_r[e]; 256 threads =
// 32 tokens x 8 column groups.
__global__ void __launch_bounds__(256) dispatch_bwd_dense_kernel(
    const uint4* __restrict__ dxd, const int32_t* __restrict__ slot_of_route,
    const float* __restrict__ dlogits, const __nv_bfloat16* __restrict__ w_router, int T, int d,
    int E, int k, uint4* __restrict__ dx) {
  pdl_begin();
  __shared__ __align__(16) __nv_bfloat16 s_w[kDenseE][kDenseCols];
  __shared__ float s_dl[kDenseTok][kDenseE + 1];
  const int tl = threadIdx.x >> 3;
  const int cg = threadIdx.x & 7;
  const int t = blockIdx.x * kDenseTok + tl;
  const int c0 = blockIdx.y * kDenseCols;
  const int nv = d / 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int slot = slot_of_route[(size_t)t * k + j];
      float f[8];
      uint4 vv = make_uint4(0, 0, 0, 0);
      MOE_CHECKED(slot, rows_max_of(T, k, E)) vv = __ldg(dxd + (size_t)slot * nv + c0 / 8 + cg);
      unpack8(vv, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
  }
  for (int e0 = 0; e0 < E; e0 += kDenseE) {
    const int ne = min(kDenseE, E - e0);
    __syncthreads();
    // W_r rows e0.., columns c0..c0+64: 16 bytes per thread and pass
    for (int i = threadIdx.x; i < ne * 8; i += blockDim.x) {
      const int r = i >> 3, q = i & 7;
      *reinterpret_cast<uint4*>(&s_w[r][q * 8]) =
          __ldg(reinterpret_cast<const uint4*>(w_router + (size_t)(e0 + r) * d + c0) + q);
    }
    for (int i = threadIdx.x; i < kDenseTok * ne; i += blockDim.x) {
      const int r = i / ne, e = i - r * ne;
      const int tt = blockIdx.x * kDenseTok + r;
      s_dl[r][e] = (tt < T) ? dlogits[(size_t)tt * E + e0 + e] : 0.0f;
    }
    __syncthreads();
    for (int e = 0; e < ne; ++e) {
      const float g = s_dl[tl][e];
      float w[8];
      unpack8(*reinterpret_cast<const uint4*>(&s_w[e][cg * 8]), w);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, w[i], acc[i]);
    }
  }
  if (t < T) dx[(size_t)t * nv + c0 / 8 + cg] = pack8(acc);
}

// partial[s][e][c] = sum over the tokens of split s of dlogits[t, e] x[t][c];
// grid (d / 64, splits), 256 threads = 32 experts x 8 column groups, token
// sub-chunks of 64 staged in shared memory.
constexpr int kDwTok = 64;
__global__ void __launch_bounds__(256) router_bwd_dense_partial_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ dlogits, int T, int d, int E,
    int splits, float* __restrict__ partial) {
  pdl_begin();
  __shared__ __align__(16) __nv_bfloat16 s_x[kDwTok][kDenseCols];
  __shared__ float s_dl[kDwTok][33];
  const int el = threadIdx.x >> 3;   // expert within the 32-expert chunk
  const int cg = threadIdx.x & 7;
  const int c0 = blockIdx.x * kDenseCols;
  const int per = (T + splits - 1) / splits;
  const int tb = blockIdx.y * per;
  const int te = min(T, tb + per);
  for (int e0 = 0; e0 < E; e0 += 32) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int t0 = tb; t0 < te; t0 += kDwTok) {
      const int nt = min(kDwTok, te - t0);
      __syncthreads();
      for (int i = threadIdx.x; i < nt * 8; i += blockDim.x) {
        const int r = i >> 3, q = i & 7;
        *reinterpret_cast<uint4*>(&s_x[r][q * 8]) =
            __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * d + c0) + q);
      }
      for (int i = threadIdx.x; i < nt * 32; i += blockDim.x) {
        const int r = i >> 5, e = i & 31;
        s_dl[r][e] = (e0 + e < E) ? dlogits[(size_t)(t0 + r) * E + e0 + e] : 0.0f;
      }
      __syncthreads();
      for (int r = 0; r < nt; ++r) {
        const float g = s_dl[r][el];
        float xv[8];
        unpack8(*reinterpret_cast<const uint4*>(&s_x[r][cg * 8]), xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, xv[i], acc[i]);
      }
    }
    if (e0 + el < E) {
      float4* dst = reinterpret_cast<float4*>(
          partial + ((size_t)blockIdx.y * E + e0 + el) * d + c0 + cg * 8);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

// dW_r[e][c] = sum over splits in order.
__global__ void __launch_bounds__(256) router_bwd_dense_reduce_kernel(
    const float* __restrict__ partial, int splits, int64_t n, float* __restrict__ dw) {
  pdl_begin();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = 0.0f;
  for (int sp = 0; sp < splits; ++sp) s += partial[(size_t)sp * n + i];
  dw[i] = s;
}

}  // namespace

int lb_partial_blocks(int T) { return (T + kLbTokensPerBlock - 1) / kLbTokensPerBlock; }

cudaError_t launch_load_balance(const float* logits, const int32_t* counts, int T, int E, int k,
                                float* partial, float* lb_stats, cudaStream_t s) {
  const int nb = lb_partial_blocks(T);
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    launch_pdl(lb_partial_kernel<1>, dim3(nb), dim3(256), 0, s, logits, T, E, partial);
  else if (epl <= 2)
    launch_pdl(lb_partial_kernel<2>, dim3(nb), dim3(256), 0, s, logits, T, E, partial);
  else if (epl <= 4)
    launch_pdl(lb_partial_kernel<4>, dim3(nb), dim3(256), 0, s, logits, T, E, partial);
  else
    launch_pdl(lb_partial_kernel<8>, dim3(nb), dim3(256), 0, s, logits, T, E, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  launch_pdl(lb_finish_kernel, dim3(1), dim3(256), 0, s, static_cast<const float*>(partial), nb,
             counts, T, E, k, lb_stats);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_bwd_dense(const void* dxd, const int32_t* slot_of_route,
                                      const float* dlogits, const void* w_router, int T, int d,
                                      int E, int k, void* dx, cudaStream_t s) {
  dim3 grid((unsigned)((T + kDenseTok - 1) / kDenseTok), (unsigned)(d / kDenseCols));
  launch_pdl(dispatch_bwd_dense_kernel, grid, dim3(256), 0, s, static_cast<const uint4*>(dxd),
             slot_of_route, dlogits, static_cast<const __nv_bfloat16*>(w_router), T, d, E, k,
             static_cast<uint4*>(dx));
  return cudaGetLastError();
}

cudaError_t launch_router_bwd_dense(const void* x, const float* dlogits, int T, int d, int E,
                                    float* partial, float* dw_router, cudaStream_t s) {
  const int splits = router_dense_splits(E);
  dim3 grid((unsigned)(d / kDenseCols), (unsigned)splits);
  launch_pdl(router_bwd_dense_partial_kernel, grid, dim3(256), 0, s,
             static_cast<const __nv_bfloat16*>(x), dlogits, T, d, E, splits, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)E * d;
  launch_pdl(router_bwd_dense_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
             static_cast<const float*>(partial), splits, n, dw_router);
  return cudaGetLastError();
}

MOE_CHECK_WORD_ACCESSOR(balance)

}  // namespace moe
