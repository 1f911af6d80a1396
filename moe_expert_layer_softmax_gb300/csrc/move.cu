// Data-movement kernels (sm_103a), all HBM-bound, 16-byte vector accesses:
//   dispatch      x[t] -> xd[slot(t, j)] for every choice j (rowwise: each token
//                 row is written straight into its expert's contiguous buffer,
//                 "Supercharging Olmo-core for Efficient and Scalable MoE
//                 Training", Abstract) and zero padding rows;
//   combine       out[t] = sum_j g_tj y[slot(t, j)]  (fp32 sum in j order);
//   combine_bwd   d_gates, dy, dlogits;
//   dispatch_bwd  dx[t] = sum_j dxd[slot(t, j)] + sum_j dl_tj W_r[e_tj];
//   router_bwd    dW_r[e] = sum of dl * x over expert e's routes (two passes:
//                 per-tile partial sums, then a fixed-order sum over tiles).
// One warp per token row; a lane moves 8 bf16 (16 bytes) per access.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMoveThreads = 256;
constexpr int kWarpsPerBlock = kMoveThreads / 32;
constexpr int kVec = 8;  // bf16 per 16-byte vector

// Zero row `row` (d bf16) with one warp.
MOE_DEV void zero_row(uint4* base, int d, int lane) {
  const int nv = d / kVec;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int c = lane; c < nv; c += 32) base[c] = z;
}

// MXFP8 codes of an all-zero row: zero codes, every block scale 2^0 (byte 127).
MOE_DEV void zero_row_mx(uint8_t* codes, uint8_t* scales, int64_t row, int d, int lane) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int c = lane; c < d / 16; c += 32) reinterpret_cast<uint4*>(codes)[c] = z;
  for (int b = lane; b < d / 32; b += 32) scales[sf_offset(row, b, d / 32)] = 127;
}

// Padding rows of expert e: [128*tile_off[e] + counts[e], 128*tile_off[e+1]).
// `p` enumerates E*128 candidates; returns the row or -1.
MOE_DEV int pad_row(int p, const int32_t* counts, const int32_t* tile_offsets) {
  const int e = p / kTileM;
  const int q = p % kTileM;
  const int row = tile_offsets[e] * kTileM + counts[e] + q;
  return (row < tile_offsets[e + 1] * kTileM) ? row : -1;
}

__global__ void __launch_bounds__(kMoveThreads) dispatch_bf16_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ slot_of_route,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ tile_offsets, int T, int d,
    int E, int k, int token_blocks, uint4* __restrict__ xd) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int nv = d / kVec;
  if (blockIdx.x < token_blocks) {
    const int t = w;
    if (t >= T) return;
    const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
    const uint4* src = x + (size_t)t * nv;
    for (int c0 = 0; c0 < nv; c0 += 32 * 4) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nv) v[u] = __ldg(src + c);
      }
      for (int j = 0; j < k; ++j) {
        const int slot = __shfl_sync(0xffffffffu, my_slot, j);
        uint4* dst = xd + (size_t)slot * nv;
        MOE_CHECKED(slot, rows_max_of(T, k, E)) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nv) dst[c] = v[u];
          }
        }
      }
    }
  } else {
    const int p = (blockIdx.x - token_blocks) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (p >= E * kTileM) return;
    const int row = pad_row(p, counts, tile_offsets);
    if (row >= 0) MOE_CHECKED(row, rows_max_of(T, k, E)) zero_row(xd + (size_t)row * nv, d, lane);
  }
}

__global__ void __launch_bounds__(kMoveThreads) combine_kernel(
    const uint4* __restrict__ y, const float* __restrict__ gates,
    const int32_t* __restrict__ slot_of_route, int T, int d, int E, int k, uint4* __restrict__ out) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int nv = d / kVec;
  const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
  const float my_g = (lane < k) ? gates[(size_t)t * k + lane] : 0.0f;
  // the column loop is warp-uniform (shuffles inside); lanes past the row end
  // read column 0 and do not store
  for (int c0 = 0; c0 < nv; c0 += 32) {
    const int c = c0 + lane;
    const bool ok = c < nv;
    const int cc = ok ? c : 0;
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
    int j = 0;
    for (; j + 4 <= k; j += 4) {
      uint4 v[4];
      float g[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int slot = __shfl_sync(0xffffffffu, my_slot, j + u);
        g[u] = __shfl_sync(0xffffffffu, my_g, j + u);
        uint4 vv = make_uint4(0, 0, 0, 0);
        MOE_CHECKED(slot, rows_max_of(T, k, E)) vv = __ldg(y + (size_t)slot * nv + cc);
        v[u] = vv;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f[kVec];
        unpack8(v[u], f);
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = fmaf(g[u], f[i], acc[i]);
      }
    }
    for (; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      float f[kVec];
      uint4 vv = make_uint4(0, 0, 0, 0);
      MOE_CHECKED(slot, rows_max_of(T, k, E)) vv = __ldg(y + (size_t)slot * nv + cc);
      unpack8(vv, f);
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[i] = fmaf(g, f[i], acc[i]);
    }
    if (ok) out[(size_t)t * nv + c] = pack8(acc);
  }
}

// KM = compile-time bound on k (4 and 8 cover the workloads; 32 is the generic
// fallback).  Per 256-column chunk a lane loads dOut once and the k rows of y
// together, so k + 1 16-byte loads are in flight per lane.  With dyq non-null
// every dy row is also quantised to MXFP8 along d (the bf16 values stored in
// dy, 32 per block: four lanes' vectors), exactly as the row quantiser would.
template <int KM>
__global__ void __launch_bounds__(kMoveThreads, KM <= 4 ? 4 : (KM <= 8 ? 3 : 1)) combine_bwd_kernel(
    const uint4* __restrict__ d_out, const uint4* __restrict__ y, const float* __restrict__ gates,
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot_of_route,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ tile_offsets, int T, int d,
    int E, int k, int token_blocks, uint4* __restrict__ dy, uint8_t* __restrict__ dyq,
    uint8_t* __restrict__ dys, float* __restrict__ d_gates, float* __restrict__ dlogits,
    const float* __restrict__ lb_logits, float lb_scale) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int nv = d / kVec;
  if (blockIdx.x >= token_blocks) {
    const int p = (blockIdx.x - token_blocks) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (p >= E * kTileM) return;
    const int row = pad_row(p, counts, tile_offsets);
    if (row >= 0) MOE_CHECKED(row, rows_max_of(T, k, E)) {
      zero_row(dy + (size_t)row * nv, d, lane);
      if (dyq != nullptr) zero_row_mx(dyq + (size_t)row * d, dys, row, d, lane);
    }
    return;
  }
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
  const float my_g = (lane < k) ? gates[(size_t)t * k + lane] : 0.0f;
  const int my_id = (lane < k) ? topk_idx[(size_t)t * k + lane] : 0;
  int slot[KM];
  float g[KM], part[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    slot[j] = __shfl_sync(0xffffffffu, my_slot, j < k ? j : 0);
    g[j] = __shfl_sync(0xffffffffu, my_g, j < k ? j : 0);
    part[j] = 0.0f;
  }
  const uint4* dO = d_out + (size_t)t * nv;
  // d is a multiple of 128 (nv of 16): the four lanes of a 32-column block are
  // all in range or all out of it, and every lane takes part in the shuffles
  for (int c0 = 0; c0 < nv; c0 += 32) {      // warp-uniform
    const int c = c0 + lane;
    const bool act = c < nv;
    float a[kVec];
    unpack8(act ? __ldg(dO + c) : make_uint4(0, 0, 0, 0), a);
    uint4 yv[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      yv[j] = make_uint4(0, 0, 0, 0);
      const int sj = KM > 8 ? __shfl_sync(0xffffffffu, my_slot, j < k ? j : 0) : slot[j];
      if (j < k && act) MOE_CHECKED(sj, rows_max_of(T, k, E)) yv[j] = __ldg(y + (size_t)sj * nv + c);
    }
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        float b[kVec];
        unpack8(yv[j], b);
#pragma unroll
        for (int i = 0; i < kVec; ++i) part[j] = fmaf(a[i], b[i], part[j]);
      }
    }
    // the k dy rows (g_j dOut[t]) once the y rows are no longer held
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        // k > 8: the route's slot and gate from the lane that holds them
        const int sj = KM > 8 ? __shfl_sync(0xffffffffu, my_slot, j) : slot[j];
        const float gj = KM > 8 ? __shfl_sync(0xffffffffu, my_g, j) : g[j];
        float o[kVec];
#pragma unroll
        for (int i = 0; i < kVec; ++i) o[i] = gj * a[i];
        const uint4 ob = pack8(o);
        if (act) MOE_CHECKED(sj, rows_max_of(T, k, E)) dy[(size_t)sj * nv + c] = ob;
        if (dyq != nullptr) {   // warp-uniform
          float q[kVec];
          unpack8(ob, q);
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < kVec; ++i) amax = fmaxf(amax, fabsf(q[i]));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          const int sx = mx_scale_exp(amax);
          const float inv = exp2i(-sx);
#pragma unroll
          for (int i = 0; i < kVec; ++i) q[i] *= inv;
          const uint2 code = e4m3x8(q);
          if (act) MOE_CHECKED(sj, rows_max_of(T, k, E)) {
            reinterpret_cast<uint2*>(dyq + (size_t)sj * d)[c] = code;
            if ((lane & 3) == 0) dys[sf_offset(sj, c / 4, d / 32)] = (uint8_t)(sx + 127);
          }
        }
      }
    }
  }
  float my_dg = 0.0f;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    if (j < k) {
      float v = part[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == j) my_dg = v;
    }
  }
  // dl_j = g_j (dg_j - sum_i g_i dg_i) on the selected experts
  float inner = (lane < k) ? my_g * my_dg : 0.0f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) inner += __shfl_xor_sync(0xffffffffu, inner, off);
  const float my_dl = my_g * (my_dg - inner);
  if (lane < k) d_gates[(size_t)t * k + lane] = my_dg;
  if (dlogits != nullptr) {
    // load-balancing term (lb_scale = coef * E / T): every logit gets
    // lb_scale * p_e (f_e - sum_e' f_e' p_e'), f_e = counts[e] / (T k)
    float lb_max = -INFINITY, lb_z = 0.0f, lb_s = 0.0f;
    const float inv_rk = 1.0f / ((float)T * (float)k);
    if (lb_scale != 0.0f) {
      const float* row = lb_logits + (size_t)t * E;
      for (int e0 = 0; e0 < E; e0 += 32)
        if (e0 + lane < E) lb_max = fmaxf(lb_max, __ldg(row + e0 + lane));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        lb_max = fmaxf(lb_max, __shfl_xor_sync(0xffffffffu, lb_max, off));
      for (int e0 = 0; e0 < E; e0 += 32) {
        if (e0 + lane < E) {
          const float pe = expf(__ldg(row + e0 + lane) - lb_max);
          lb_z += pe;
          lb_s += pe * ((float)counts[e0 + lane] * inv_rk);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        lb_z += __shfl_xor_sync(0xffffffffu, lb_z, off);
        lb_s += __shfl_xor_sync(0xffffffffu, lb_s, off);
      }
      lb_s /= lb_z;
    }
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      float v = 0.0f;
      for (int j = 0; j < k; ++j) {
        const int id = __shfl_sync(0xffffffffu, my_id, j);
        const float dl = __shfl_sync(0xffffffffu, my_dl, j);
        if (id == e) v = dl;
      }
      if (lb_scale != 0.0f && e < E) {
        const float pe = expf(__ldg(lb_logits + (size_t)t * E + e) - lb_max) / lb_z;
        v += lb_scale * pe * ((float)counts[e] * inv_rk - lb_s);
      }
      if (e < E) dlogits[(size_t)t * E + e] = v;
    }
  }
}

template <int KM>
__global__ void __launch_bounds__(kMoveThreads, KM <= 4 ? 4 : (KM <= 8 ? 3 : 1)) dispatch_bwd_kernel(
    const uint4* __restrict__ dxd, const int32_t* __restrict__ slot_of_route,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ dlogits,
    const uint4* __restrict__ w_router, int T, int d, int E, int k, uint4* __restrict__ dx) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int nv = d / kVec;
  const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
  const int my_id = (lane < k) ? topk_idx[(size_t)t * k + lane] : 0;
  const float my_dl =
      (lane < k && w_router != nullptr) ? dlogits[(size_t)t * E + my_id] : 0.0f;
  int slot[KM], id[KM];
  float dl[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    const int src = j < k ? j : 0;
    slot[j] = __shfl_sync(0xffffffffu, my_slot, src);
    id[j] = __shfl_sync(0xffffffffu, my_id, src);
    dl[j] = __shfl_sync(0xffffffffu, my_dl, src);
  }
  // two 32-vector column chunks per pass (KM <= 8): the k rows of both chunks
  // are loaded before any is used, 2k 16-byte loads in flight per lane
  constexpr int kCh = KM <= 8 ? 2 : 1;
  for (int c0 = 0; c0 < nv; c0 += 32 * kCh) {
    uint4 v[kCh][KM];
#pragma unroll
    for (int h = 0; h < kCh; ++h) {
      const int c = c0 + 32 * h + lane;
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        v[h][j] = make_uint4(0, 0, 0, 0);
        if (j < k && c < nv)
          MOE_CHECKED(slot[j], rows_max_of(T, k, E)) v[h][j] = __ldg(dxd + (size_t)slot[j] * nv + c);
      }
    }
#pragma unroll
    for (int h = 0; h < kCh; ++h) {
      const int c = c0 + 32 * h + lane;
      if (c >= nv) continue;
      float acc[kVec];
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        if (j < k) {
          float f[kVec];
          unpack8(v[h][j], f);
#pragma unroll
          for (int i = 0; i < kVec; ++i) acc[i] += f[i];
        }
      }
      if (w_router != nullptr) {
        uint4 w[KM];
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          w[j] = make_uint4(0, 0, 0, 0);
          if (j < k) MOE_CHECKED(id[j], E) w[j] = __ldg(w_router + (size_t)id[j] * nv + c);
        }
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (j < k) {
            float f[kVec];
            unpack8(w[j], f);
#pragma unroll
            for (int i = 0; i < kVec; ++i) acc[i] = fmaf(dl[j], f[i], acc[i]);
          }
        }
      }
      dx[(size_t)t * nv + c] = pack8(acc);
    }
  }
}

// k > 8 (up to 32 routes per token): the route's slot, expert and dlogit come
// from the lane that holds them, and the rows are loaded 8 routes at a time
// (8 16-byte loads in flight per lane); same sums, in route order, as above.
__global__ void __launch_bounds__(kMoveThreads) dispatch_bwd_wide_kernel(
    const uint4* __restrict__ dxd, const int32_t* __restrict__ slot_of_route,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ dlogits,
    const uint4* __restrict__ w_router, int T, int d, int E, int k, uint4* __restrict__ dx) {
  pdl_begin();
  constexpr int G = 8;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  const int nv = d / kVec;
  const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
  const int my_id = (lane < k) ? topk_idx[(size_t)t * k + lane] : 0;
  const float my_dl =
      (lane < k && w_router != nullptr) ? dlogits[(size_t)t * E + my_id] : 0.0f;
  for (int c0 = 0; c0 < nv; c0 += 32) {     // warp-uniform
    const int c = c0 + lane;
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += G) {
      uint4 v[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int j = j0 + g;
        const int sj = __shfl_sync(0xffffffffu, my_slot, j < k ? j : 0);
        v[g] = make_uint4(0, 0, 0, 0);
        if (j < k && c < nv)
          MOE_CHECKED(sj, rows_max_of(T, k, E)) v[g] = __ldg(dxd + (size_t)sj * nv + c);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (j0 + g < k) {
          float f[kVec];
          unpack8(v[g], f);
#pragma unroll
          for (int i = 0; i < kVec; ++i) acc[i] += f[i];
        }
      }
    }
    if (w_router != nullptr) {
      for (int j0 = 0; j0 < k; j0 += G) {
        uint4 w[G];
        float dlj[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int j = j0 + g;
          const int ij = __shfl_sync(0xffffffffu, my_id, j < k ? j : 0);
          dlj[g] = __shfl_sync(0xffffffffu, my_dl, j < k ? j : 0);
          w[g] = make_uint4(0, 0, 0, 0);
          if (j < k && c < nv) MOE_CHECKED(ij, E) w[g] = __ldg(w_router + (size_t)ij * nv + c);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (j0 + g < k) {
            float f[kVec];
            unpack8(w[g], f);
#pragma unroll
            for (int i = 0; i < kVec; ++i) acc[i] = fmaf(dlj[g], f[i], acc[i]);
          }
        }
      }
    }
    if (c < nv) dx[(size_t)t * nv + c] = pack8(acc);
  }
}

// Pass 1: partial[m][col] = sum over the real rows s of tile m of
// dlogits[t(s), e(m)] * x[t(s)][col], for a 1024-column chunk: 128 column
// threads x 8 columns, and four row groups (rows g, g + 4, g + 8, ...) whose
// sums are added in a fixed order at the end.  Eight row loads are in flight
// per thread.
constexpr int kRbCols = 128;
constexpr int kRbGroups = 4;
constexpr int kRbThreads = kRbGroups * kRbCols;
__global__ void __launch_bounds__(kRbThreads) router_bwd_partial_kernel(
    const uint4* __restrict__ x, const float* __restrict__ dlogits,
    const int32_t* __restrict__ route_of_slot, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ tile_offsets, int T, int d, int E, int k,
    float* __restrict__ partial) {
  pdl_begin();
  __shared__ int32_t s_tok[kTileM];
  __shared__ float s_dl[kTileM];
  __shared__ float4 s_odd[kRbGroups - 1][2][kRbCols];
  const int m = blockIdx.x;
  if (m >= tile_offsets[E]) return;
  // expert owning tile m: the largest e with tile_offsets[e] <= m
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_offsets[mid] <= m) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int nv = d / kVec;
  const int row_end = tile_offsets[e] * kTileM + counts[e];
  const int r0 = m * kTileM;
  const int nrows = max(0, min(kTileM, row_end - r0));
  if (threadIdx.x < nrows) {
    int t = 0;
    float dl = 0.0f;
    MOE_CHECKED(r0 + threadIdx.x, rows_max_of(T, k, E)) {
      const int tt = route_of_slot[r0 + threadIdx.x] / k;
      MOE_CHECKED(tt, T) {
        t = tt;
        dl = dlogits[(size_t)tt * E + e];
      }
    }
    s_tok[threadIdx.x] = t;
    s_dl[threadIdx.x] = dl;
  }
  __syncthreads();
  const int ct = threadIdx.x % kRbCols;
  const int grp = threadIdx.x / kRbCols;        // rows grp, grp + G, grp + 2G, ...
  const int c = blockIdx.y * kRbCols + ct;
  const bool ok = c < nv;
  float acc[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
  if (ok) {
    int r = grp;
    for (; r + 7 * kRbGroups < nrows; r += 8 * kRbGroups) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldg(x + (size_t)s_tok[r + kRbGroups * u] * nv + c);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float f[kVec];
        unpack8(v[u], f);
        const float dl = s_dl[r + kRbGroups * u];
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = fmaf(dl, f[i], acc[i]);
      }
    }
    for (; r < nrows; r += kRbGroups) {
      float f[kVec];
      unpack8(__ldg(x + (size_t)s_tok[r] * nv + c), f);
      const float dl = s_dl[r];
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[i] = fmaf(dl, f[i], acc[i]);
    }
  }
  if (grp > 0) {
    s_odd[grp - 1][0][ct] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    s_odd[grp - 1][1][ct] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncthreads();
  if (grp == 0 && ok) {
#pragma unroll
    for (int g2 = 0; g2 < kRbGroups - 1; ++g2) {
      const float4 a = s_odd[g2][0][ct], b = s_odd[g2][1][ct];
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    float4* dst = reinterpret_cast<float4*>(partial + (size_t)m * d + (size_t)c * kVec);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Pass 2: dW_r[e][col] = sum over e's tiles in order (zero for empty experts).
__global__ void __launch_bounds__(256) router_bwd_reduce_kernel(
    const float* __restrict__ partial, const int32_t* __restrict__ tile_offsets, int d,
    float* __restrict__ dw) {
  pdl_begin();
  const int e = blockIdx.y;
  const int col = blockIdx.x * 256 + threadIdx.x;
  if (col >= d) return;
  float s = 0.0f;
  for (int m = tile_offsets[e]; m < tile_offsets[e + 1]; ++m) s += partial[(size_t)m * d + col];
  dw[(size_t)e * d + col] = s;
}

int pad_blocks(int E) { return (E * kTileM + kWarpsPerBlock - 1) / kWarpsPerBlock; }

}  // namespace

cudaError_t launch_dispatch_bf16(const void* x, const int32_t* slot_of_route,
                                 const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                                 int E, int k, void* xd, cudaStream_t s) {
  const int tb = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  launch_pdl(dispatch_bf16_kernel, dim3(tb + pad_blocks(E)), dim3(kMoveThreads), 0, s, 
      static_cast<const uint4*>(x), slot_of_route, counts, tile_offsets, T, d, E, k, tb,
      static_cast<uint4*>(xd));
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const float* gates, const int32_t* slot_of_route, int T,
                           int d, int E, int k, void* out, cudaStream_t s) {
  const int tb = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  launch_pdl(combine_kernel, dim3(tb), dim3(kMoveThreads), 0, s, static_cast<const uint4*>(y), gates, slot_of_route, T,
                                             d, E, k, static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const void* d_out, const void* y, const float* gates,
                               const int32_t* topk_idx, const int32_t* slot_of_route,
                               const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                               int E, int k, void* dy, float* d_gates, float* dlogits,
                               cudaStream_t s, const float* lb_logits, float lb_scale,
                               uint8_t* dyq, uint8_t* dys) {
  const int tb = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (k <= 4)
    launch_pdl(combine_bwd_kernel<4>, dim3(tb + pad_blocks(E)), dim3(kMoveThreads), 0, s,
        static_cast<const uint4*>(d_out), static_cast<const uint4*>(y), gates, topk_idx,
        slot_of_route, counts, tile_offsets, T, d, E, k, tb, static_cast<uint4*>(dy), dyq, dys,
        d_gates, dlogits, lb_logits, lb_scale);
  else if (k <= 8)
    launch_pdl(combine_bwd_kernel<8>, dim3(tb + pad_blocks(E)), dim3(kMoveThreads), 0, s, 
        static_cast<const uint4*>(d_out), static_cast<const uint4*>(y), gates, topk_idx,
        slot_of_route, counts, tile_offsets, T, d, E, k, tb, static_cast<uint4*>(dy), dyq, dys,
        d_gates, dlogits, lb_logits, lb_scale);
  else
    launch_pdl(combine_bwd_kernel<32>, dim3(tb + pad_blocks(E)), dim3(kMoveThreads), 0, s, 
        static_cast<const uint4*>(d_out), static_cast<const uint4*>(y), gates, topk_idx,
        slot_of_route, counts, tile_offsets, T, d, E, k, tb, static_cast<uint4*>(dy), dyq, dys,
        d_gates, dlogits, lb_logits, lb_scale);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_bwd(const void* dxd, const int32_t* slot_of_route,
                                const int32_t* topk_idx, const float* dlogits,
                                const void* w_router, int T, int d, int E, int k, void* dx,
                                cudaStream_t s) {
  const int tb = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (k <= 4)
    launch_pdl(dispatch_bwd_kernel<4>, dim3(tb), dim3(kMoveThreads), 0, s,
        static_cast<const uint4*>(dxd), slot_of_route, topk_idx, dlogits,
        static_cast<const uint4*>(w_router), T, d, E, k, static_cast<uint4*>(dx));
  else if (k <= 8)
    launch_pdl(dispatch_bwd_kernel<8>, dim3(tb), dim3(kMoveThreads), 0, s, 
        static_cast<const uint4*>(dxd), slot_of_route, topk_idx, dlogits,
        static_cast<const uint4*>(w_router), T, d, E, k, static_cast<uint4*>(dx));
  else
    launch_pdl(dispatch_bwd_wide_kernel, dim3(tb), dim3(kMoveThreads), 0, s,
        static_cast<const uint4*>(dxd), slot_of_route, topk_idx, dlogits,
        static_cast<const uint4*>(w_router), T, d, E, k, static_cast<uint4*>(dx));
  return cudaGetLastError();
}

cudaError_t launch_router_bwd(const void* x, const float* dlogits, const int32_t* route_of_slot,
                              const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                              int E, int k, int64_t tiles_max, float* partial, float* dw_router,
                              cudaStream_t s) {
  (void)T;
  const int nv = d / kVec;
  dim3 g1((unsigned)tiles_max, (unsigned)((nv + kRbCols - 1) / kRbCols));
  launch_pdl(router_bwd_partial_kernel, dim3(g1), dim3(kRbThreads), 0, s, static_cast<const uint4*>(x), dlogits,
                                                      route_of_slot, counts, tile_offsets, T, d, E, k,
                                                      partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((unsigned)((d + 255) / 256), (unsigned)E);
  launch_pdl(router_bwd_reduce_kernel, dim3(g2), dim3(256), 0, s, partial, tile_offsets, d, dw_router);
  return cudaGetLastError();
}

MOE_CHECK_WORD_ACCESSOR(move)

}  // namespace moe
