// Routing kernels (sm_103a): warp-shuffle softmax/top-k with renormalised gates,
// per-block expert histograms with stable in-block ranks, the counts/offsets
// scan, and the slot maps.  All routing metadata stays on the device
// ("Supercharging Olmo-core for Efficient and Scalable MoE Training", Abstract;
// Section 24.1: the device-resident metadata removes the host wait without
// changing the routing calculation).
//
// Determinism: a route's slot is (base of its block for its expert) + (its rank
// among the block's routes of that expert, in (token, choice) order), and the
// block bases are a scan over blocks in block order.  This is exactly the
// sequential walk over routes in ascending (t, j) order, independent of timing.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTopkThreads = 256;  // 8 warps; each warp handles 2 of the block's 16 tokens

// Order used for the selection: larger key first, lower expert id on ties.
// NaN is treated as -inf so that the selection stays a valid set of k distinct
// experts; the token is flagged and its gates are zeroed.
MOE_DEV float route_key(float v) { return (v != v) ? -CUDART_INF_F : v; }

template <int EPL>
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ int32_t s_sel[kRouteTokensPerBlock * 32];  // expert of each route of the block
  __shared__ int32_t s_cnt[256];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kRouteTokensPerBlock;
  const int ntok = min(kRouteTokensPerBlock, T - t0);

  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;

  for (int tl = warp; tl < ntok; tl += kTopkThreads / 32) {
    const int t = t0 + tl;
    const float* row = logits + (size_t)t * E;
    float key[EPL];
    uint32_t taken = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      float v = (e < E) ? __ldg(row + e) : 0.0f;
      if (e < E && !isfinite(v)) bad = true;
      key[i] = route_key(v);
      if (e >= E) taken |= 1u << i;
    }
    const bool token_bad = __any_sync(0xffffffffu, bad);

    float my_val = 0.0f, lmax = 0.0f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float bv = 0.0f;
      int bid = -1;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (!(taken & (1u << i)) && (bid < 0 || key[i] > bv)) {
          bv = key[i];
          bid = lane + 32 * i;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oid = __shfl_xor_sync(0xffffffffu, bid, off);
        if (oid >= 0 && (bid < 0 || ov > bv || (ov == bv && oid < bid))) {
          bv = ov;
          bid = oid;
        }
      }
      if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
      if (j == 0) lmax = bv;
      if (lane == j) {
        my_val = bv;
        my_id = bid;
      }
      if (lane == 0) s_sel[tl * k + j] = bid;
    }
    // gates: softmax over the k selected logits (equal to the full softmax
    // renormalised over the selection)
    float ex = (lane < k) ? expf(my_val - lmax) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_id;
      gates[(size_t)t * k + lane] = token_bad ? 0.0f : ex / sum;
    }
    if (token_bad && lane == 0) raise_error(err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();

  // Stable ranks of the block's routes within their experts, in route order.
  if (warp == 0) {
    const int n = ntok * k;
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < n; base += 32) {
      const int r = base + lane;
      const bool active = r < n;
      const uint32_t act = __ballot_sync(0xffffffffu, active);
      if (active) {
        const int e = s_sel[r];
        const uint32_t peers = __match_any_sync(act, e);
        const int rank = s_cnt[e] + __popc(peers & lt_mask);
        local_rank[(size_t)t0 * k + r] = rank;
        __syncwarp(act);
        if ((__ffs(peers) - 1) == lane) s_cnt[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) block_hist[(size_t)blockIdx.x * E + e] = s_cnt[e];
}

// One block of 1024 threads.  Thread (p, e) = (tid / Epad, tid % Epad) owns
// expert e and the p-th contiguous chunk of the top-k blocks.  block_hist[b][e]
// (routes of expert e in block b) is replaced by the absolute first row of
// block b's routes of e; counts, offsets and tile_offsets are written.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(kScanThreads) route_scan_kernel(
    int32_t* __restrict__ block_hist, int n_blocks, int E, int e_pad,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ tile_offsets) {
  pdl_begin();
  __shared__ int32_t s_part[kScanThreads];  // [p][e] chunk sums
  __shared__ int32_t s_c[256];
  __shared__ int32_t s_t[256];
  const int tid = threadIdx.x;
  const int e = tid % e_pad;
  const int p = tid / e_pad;
  const int P = kScanThreads / e_pad;
  const int cb = (n_blocks + P - 1) / P;
  const int b0 = min(n_blocks, p * cb);
  const int b1 = min(n_blocks, b0 + cb);
  int sum = 0;
  if (e < E)
    for (int b = b0; b < b1; ++b) sum += block_hist[(size_t)b * E + e];
  s_part[tid] = sum;
  __syncthreads();
  int prefix = 0, total = 0;
  if (e < E) {
    for (int q = 0; q < P; ++q) {
      const int v = s_part[q * e_pad + e];
      prefix += (q < p) ? v : 0;
      total += v;
    }
  }
  if (tid < 256) {
    s_c[tid] = 0;
    s_t[tid] = 0;
  }
  __syncthreads();
  if (p == 0 && e < E) {
    s_c[e] = total;
    s_t[e] = (total + kTileM - 1) / kTileM;
  }
  __syncthreads();
  // inclusive Hillis-Steele scans over 256 entries (threads 0..255)
  for (int off = 1; off < 256; off <<= 1) {
    int c = 0, t = 0;
    if (tid < 256 && tid >= off) {
      c = s_c[tid - off];
      t = s_t[tid - off];
    }
    __syncthreads();
    if (tid < 256) {
      s_c[tid] += c;
      s_t[tid] += t;
    }
    __syncthreads();
  }
  if (e < E) {
    const int tiles = (total + kTileM - 1) / kTileM;
    if (p == 0) {
      counts[e] = total;
      offsets[e + 1] = s_c[e];
      tile_offsets[e + 1] = s_t[e];
    }
    int base = (s_t[e] - tiles) * kTileM + prefix;
    for (int b = b0; b < b1; ++b) {
      const int h = block_hist[(size_t)b * E + e];
      block_hist[(size_t)b * E + e] = base;
      base += h;
    }
  }
  if (tid == 0) {
    offsets[0] = 0;
    tile_offsets[0] = 0;
  }
}

__global__ void __launch_bounds__(256) route_slots_kernel(
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ local_rank,
    const int32_t* __restrict__ block_base, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ tile_offsets, int T, int E, int k, int64_t rows_max,
    int32_t* __restrict__ slot_of_route, int32_t* __restrict__ route_of_slot,
    int32_t* __restrict__ err) {
  pdl_begin();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t R = (int64_t)T * k;
  if (i < R) {
    const int t = (int)(i / k);
    const int b = t / kRouteTokensPerBlock;
    const int e = topk_idx[i];
    const int slot = (e >= 0 && e < E) ? block_base[(size_t)b * E + e] + local_rank[i] : -1;
    if (slot < 0 || slot >= rows_max) {   // never expected
      raise_error(err, MOE_DEVERR_BOUNDS);
      slot_of_route[i] = 0;
      return;
    }
    slot_of_route[i] = slot;
    route_of_slot[slot] = (int32_t)i;
  } else if (i < R + (int64_t)E * kTileM) {
    const int p = (int)(i - R);
    const int e = p / kTileM;
    const int q = p % kTileM;
    const int row = tile_offsets[e] * kTileM + counts[e] + q;
    if (row < tile_offsets[e + 1] * kTileM) route_of_slot[row] = -1;
  }
}

// Scan and slots in one kernel.  Block b < n_route_blk handles the routes of
// routing blocks [4b, 4b + 4) (64 tokens); the blocks after them mark the
// padding rows.  Every block re-derives from the per-block histograms (read
// only, L2-resident) the per-expert totals and tile offsets, and a route block
// the prefix over the routing blocks before its own; block 0 writes counts,
// offsets and tile_offsets.  The slots are those of the sequential walk over
// routes in (t, j) order, as with the separate scan and slots kernels.
constexpr int kSsThreads = 256;
constexpr int kSsRouteBlocks = 4;   // routing blocks (16 tokens each) per block
__global__ void __launch_bounds__(kSsThreads) route_scan_slots_kernel(
    const int32_t* __restrict__ block_hist, int n_blocks, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ local_rank, int T, int E, int k, int64_t rows_max,
    int n_route_blk, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ tile_offsets, int32_t* __restrict__ slot_of_route,
    int32_t* __restrict__ route_of_slot, int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ int32_t s_ptot[4 * kSsThreads];   // [part][expert] partial sums
  __shared__ int32_t s_ppre[4 * kSsThreads];
  __shared__ int32_t s_c[256];                   // counts, then their inclusive scan
  __shared__ int32_t s_t[256];                   // tiles, then their inclusive scan
  __shared__ int32_t s_pre[256];
  __shared__ int32_t s_tot[256];
  __shared__ int32_t s_base[kSsRouteBlocks][256];
  const int tid = threadIdx.x;
  const bool route_blk = (int)blockIdx.x < n_route_blk;
  const int rb0 = route_blk ? (int)blockIdx.x * kSsRouteBlocks : n_blocks;

  // 1. per-expert sums over all routing blocks and over those before rb0:
  //    thread (part p, column group g) sums V experts over a range of rows
  const int V = (E % 4 == 0) ? 4 : 1;
  const int ng = E / V;
  const int P = kSsThreads / ng;
  const int p = tid / ng, g = tid - (tid / ng) * ng;
  if (p < P) {
    int tot[4] = {0, 0, 0, 0}, pre[4] = {0, 0, 0, 0};
    const int per = (n_blocks + P - 1) / P;
    const int r0 = min(n_blocks, p * per), r1 = min(n_blocks, r0 + per);
    for (int r = r0; r < r1; r += 8) {
      int4 h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        h[u] = make_int4(0, 0, 0, 0);
        if (r + u < r1) {
          const int32_t* row = block_hist + (size_t)(r + u) * E + V * g;
          if (V == 4) h[u] = *reinterpret_cast<const int4*>(row);
          else h[u].x = *row;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        tot[0] += h[u].x; tot[1] += h[u].y; tot[2] += h[u].z; tot[3] += h[u].w;
        if (r + u < rb0) {
          pre[0] += h[u].x; pre[1] += h[u].y; pre[2] += h[u].z; pre[3] += h[u].w;
        }
      }
    }
    for (int c = 0; c < V; ++c) {
      s_ptot[p * E + V * g + c] = tot[c];
      s_ppre[p * E + V * g + c] = pre[c];
    }
  }
  __syncthreads();
  if (tid < 256) {
    int tot = 0, pre = 0;
    if (tid < E)
      for (int q = 0; q < P; ++q) {
        tot += s_ptot[q * E + tid];
        pre += s_ppre[q * E + tid];
      }
    s_tot[tid] = tot;
    s_pre[tid] = pre;
    s_c[tid] = tot;
    s_t[tid] = (tot + kTileM - 1) / kTileM;
  }
  __syncthreads();
  // 2. inclusive scans of counts and tiles over 256 entries
  for (int off = 1; off < 256; off <<= 1) {
    int c = 0, t = 0;
    if (tid >= off) {
      c = s_c[tid - off];
      t = s_t[tid - off];
    }
    __syncthreads();
    s_c[tid] += c;
    s_t[tid] += t;
    __syncthreads();
  }
  if (blockIdx.x == 0 && tid < E) {
    counts[tid] = s_tot[tid];
    offsets[tid + 1] = s_c[tid];
    tile_offsets[tid + 1] = s_t[tid];
    if (tid == 0) {
      offsets[0] = 0;
      tile_offsets[0] = 0;
    }
  }
  if (!route_blk) {
    // 3'. padding rows of each expert's last tile
    const int q = ((int)blockIdx.x - n_route_blk) * kSsThreads + tid;
    if (q < E * kTileM) {
      const int e = q / kTileM;
      const int tile0 = e > 0 ? s_t[e - 1] : 0;
      const int row = tile0 * kTileM + s_tot[e] + q % kTileM;
      if (row < s_t[e] * kTileM) route_of_slot[row] = -1;
    }
    return;
  }
  // 3. first row of each of this block's routing blocks' routes, per expert
  if (tid < E) {
    int base = (s_t[tid] - (s_tot[tid] + kTileM - 1) / kTileM) * kTileM + s_pre[tid];
    for (int j = 0; j < kSsRouteBlocks; ++j) {
      s_base[j][tid] = base;
      if (rb0 + j < n_blocks) base += block_hist[(size_t)(rb0 + j) * E + tid];
    }
  }
  __syncthreads();
  // 4. the slots of this block's routes
  const int64_t i0 = (int64_t)rb0 * kRouteTokensPerBlock * k;
  const int64_t i1 = min((int64_t)T, (int64_t)(rb0 + kSsRouteBlocks) * kRouteTokensPerBlock) * k;
  for (int64_t i = i0 + tid; i < i1; i += kSsThreads) {
    const int t = (int)(i / k);
    const int j = t / kRouteTokensPerBlock - rb0;
    const int e = topk_idx[i];
    const int slot = (e >= 0 && e < E) ? s_base[j][e] + local_rank[i] : -1;
    if (slot < 0 || slot >= rows_max) {   // never expected
      raise_error(err, MOE_DEVERR_BOUNDS);
      slot_of_route[i] = 0;
      continue;
    }
    slot_of_route[i] = slot;
    route_of_slot[slot] = (int32_t)i;
  }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* gates, int32_t* local_rank, int32_t* block_hist,
                              int32_t* err, cudaStream_t s) {
  const int nb = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    launch_pdl(route_topk_kernel<1>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx, gates, local_rank,
                                                    block_hist, err);
  else if (epl <= 2)
    launch_pdl(route_topk_kernel<2>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx, gates, local_rank,
                                                    block_hist, err);
  else if (epl <= 4)
    launch_pdl(route_topk_kernel<4>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx, gates, local_rank,
                                                    block_hist, err);
  else
    launch_pdl(route_topk_kernel<8>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx, gates, local_rank,
                                                    block_hist, err);
  return cudaGetLastError();
}

cudaError_t launch_route_scan(int32_t* block_hist, int n_blocks, int E, int32_t* counts,
                              int32_t* offsets, int32_t* tile_offsets, cudaStream_t s) {
  int e_pad = 4;
  while (e_pad < E) e_pad <<= 1;   // E <= 256 -> at least 4 chunks per expert
  launch_pdl(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, block_hist, n_blocks, E, e_pad, counts, offsets,
                                               tile_offsets);
  return cudaGetLastError();
}

cudaError_t launch_route_slots(const int32_t* topk_idx, const int32_t* local_rank,
                               const int32_t* block_base, const int32_t* counts,
                               const int32_t* tile_offsets, int T, int E, int k, int64_t rows_max,
                               int32_t* slot_of_route, int32_t* route_of_slot, int32_t* err,
                               cudaStream_t s) {
  const int64_t n = (int64_t)T * k + (int64_t)E * kTileM;
  const int nb = (int)((n + 255) / 256);
  launch_pdl(route_slots_kernel, dim3(nb), dim3(256), 0, s, topk_idx, local_rank, block_base, counts, tile_offsets, T,
                                        E, k, rows_max, slot_of_route, route_of_slot, err);
  return cudaGetLastError();
}

cudaError_t launch_route_scan_slots(const int32_t* block_hist, int n_blocks,
                                    const int32_t* topk_idx, const int32_t* local_rank, int T,
                                    int E, int k, int64_t rows_max, int32_t* counts,
                                    int32_t* offsets, int32_t* tile_offsets,
                                    int32_t* slot_of_route, int32_t* route_of_slot, int32_t* err,
                                    cudaStream_t s) {
  const int n_route_blk = (n_blocks + kSsRouteBlocks - 1) / kSsRouteBlocks;
  const int n_pad_blk = (E * kTileM + kSsThreads - 1) / kSsThreads;
  launch_pdl(route_scan_slots_kernel, dim3((unsigned)(n_route_blk + n_pad_blk)), dim3(kSsThreads),
             0, s, block_hist, n_blocks, topk_idx, local_rank, T, E, k, rows_max, n_route_blk,
             counts, offsets, tile_offsets, slot_of_route, route_of_slot, err);
  return cudaGetLastError();
}

}  // namespace moe
