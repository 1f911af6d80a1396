// Routing kernels (sm_103a): warp-shuffle softmax/top-k with renormalised gates,
// per-block expert histograms with stable in-block ranks, the counts/offsets
// scan, and the slot maps.  All routing metadata stays on the device
// ("Supercharging Olmo-core for Efficient and Scalable MoE Training", Abstract;
// Section 24.1: the device-resident metadata removes the host wait without
// changing the routing calculation).
//
// Determinism: a route's slot is (base of its 128-token block for its expert) +
// (its rank among the block's routes of that expert, in (token, choice) order),
// and the block bases are a scan over blocks in block order.  This is exactly
// the sequential walk over routes in ascending (t, j) order, independent of
// timing and of which top-k kernel ran.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTpb = kRouteTokensPerBlock;   // 128 tokens per routing block

// Order used for the selection: larger key first, lower expert id on ties.
// NaN is treated as -inf so that the selection stays a valid set of k distinct
// experts; the token is flagged and its gates are zeroed.
MOE_DEV float route_key(float v) { return (v != v) ? -CUDART_INF_F : v; }

// entry (v, i) goes ahead of (w, j): larger key first, lower expert id on ties
MOE_DEV bool topk_ahead(float v, int i, float w, int j) { return v > w || (v == w && i < j); }

// gates of the k <= 8 selected keys (largest first): exp(l_j - l_1) / sum_i
// exp(l_i - l_1), the sum taken in the order of a 32-lane xor butterfly in
// which only lanes 0..k-1 are non-zero (the order route_topk_kernel uses), so
// that every top-k kernel gives the same bits
MOE_DEV float gate_sum8(const float* ex) {
  return ((ex[0] + ex[4]) + (ex[2] + ex[6])) + ((ex[1] + ex[5]) + (ex[3] + ex[7]));
}

// Ranks and histogram of one 128-token routing block from per-expert token
// masks (s_mask[4 e + w] bit b: token 32 w + b of the block chose expert e):
// a route's rank within its expert is the number of earlier tokens of the
// block with that expert, which is its place in the stable (t, j) order.
MOE_DEV int mask_rank(const uint32_t* s_mask, int e, int tl) {
  const uint32_t* mk = s_mask + 4 * e;
  int rank = __popc(mk[tl >> 5] & ((1u << (tl & 31)) - 1u));
  for (int w = 0; w < (tl >> 5); ++w) rank += __popc(mk[w]);
  return rank;
}
MOE_DEV void write_block_hist(const uint32_t* s_mask, int E, int32_t* block_hist, int tid,
                              int nthreads) {
  for (int e = tid; e < E; e += nthreads)
    block_hist[(size_t)blockIdx.x * E + e] = __popc(s_mask[4 * e]) + __popc(s_mask[4 * e + 1]) +
                                             __popc(s_mask[4 * e + 2]) + __popc(s_mask[4 * e + 3]);
}

// ---------------------------------------------------------------- top-k kernels
// (a) E <= EM <= 128, k <= 8: one thread per token with all of its logits in
// registers, k passes of argmax; a taken expert is marked in a bit mask.
template <int EM, int KM>
__global__ void __launch_bounds__(kTpb) route_topk_reg_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ uint32_t s_mask[4 * EM];
  const int tl = threadIdx.x;
  const int64_t t = (int64_t)blockIdx.x * kTpb + tl;
  const bool valid = t < T;
  for (int i = tl; i < 4 * E; i += kTpb) s_mask[i] = 0u;
  float v[EM];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < EM; ++c) v[c] = -CUDART_INF_F;   // columns >= E are never chosen (k <= E)
  if (valid) {
    const float* row = logits + t * E;
    if ((E & 3) == 0) {
#pragma unroll
      for (int c = 0; c < EM; c += 4) {
        if (c < E) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(row + c));
          v[c] = q.x; v[c + 1] = q.y; v[c + 2] = q.z; v[c + 3] = q.w;
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < EM; ++c)
        if (c < E) v[c] = __ldg(row + c);
    }
#pragma unroll
    for (int c = 0; c < EM; ++c) {
      bad = bad || !isfinite(v[c]) && c < E;
      v[c] = route_key(v[c]);
    }
  }
  uint32_t taken[EM / 32];
#pragma unroll
  for (int w = 0; w < EM / 32; ++w) taken[w] = 0u;
  int sel[KM];
  float ex[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ex[j] = 0.0f;
  float lmax = 0.0f;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    sel[j] = 0;
    if (j < k) {
      float best = 0.0f;
      int bi = -1;
#pragma unroll
      for (int c = 0; c < EM; ++c) {
        const bool free = ((taken[c >> 5] >> (c & 31)) & 1u) == 0u;
        if (free && (bi < 0 || v[c] > best)) {   // strict: the lower id keeps a tie
          best = v[c];
          bi = c;
        }
      }
#pragma unroll
      for (int w = 0; w < EM / 32; ++w)
        if ((bi >> 5) == w) taken[w] |= 1u << (bi & 31);
      sel[j] = bi;
      if (j == 0) lmax = best;
      ex[j] = expf(best - lmax);
    }
  }
  if (valid) {
    const float sum = gate_sum8(ex);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        topk_idx[t * k + j] = sel[j];
        gates[t * k + j] = bad ? 0.0f : ex[j] / sum;
      }
    }
    if (bad) raise_error(err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();   // masks cleared
  if (valid) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) atomicOr(&s_mask[4 * sel[j] + (tl >> 5)], 1u << (tl & 31));
  }
  __syncthreads();
  if (valid) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) local_rank[t * k + j] = mask_rank(s_mask, sel[j], tl);
  }
  write_block_hist(s_mask, E, block_hist, tl, kTpb);
}

// (a2) 32 < E <= 2 EH, k <= 8: two threads per token (the two lanes of a pair
// in one warp): lane h ranks experts [h EH, (h + 1) EH) in registers (k passes
// of argmax, the lower id first on ties), and both lanes merge the two sorted
// lists through shuffles of their heads - lane 0's head goes first unless lane
// 1's key is strictly larger, since lane 0 holds the lower ids - so that both
// hold the same k experts in the order of (a).  Twice the threads of (a) for
// the same tokens: the selection is latency-bound at one thread per token.
constexpr int kTopk2Threads = 2 * kTpb;
template <int EH, int KM>
__global__ void __launch_bounds__(kTopk2Threads) route_topk2_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ uint32_t s_mask[4 * 2 * EH];
  const int tid = threadIdx.x;
  const int tl = tid >> 1;              // token of the block
  const int h = tid & 1;                // which half of the experts
  const int64_t t = (int64_t)blockIdx.x * kTpb + tl;
  const bool valid = t < T;
  for (int i = tid; i < 4 * E; i += kTopk2Threads) s_mask[i] = 0u;
  const int c0 = h * EH;
  float v[EH];
  bool bad = false;
#pragma unroll
  for (int c = 0; c < EH; ++c) v[c] = -CUDART_INF_F;   // columns >= E are never chosen (k <= E)
  if (valid) {
    const float* row = logits + t * E + c0;
    if ((E & 3) == 0) {
#pragma unroll
      for (int c = 0; c < EH; c += 4) {
        if (c0 + c < E) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(row + c));
          v[c] = q.x; v[c + 1] = q.y; v[c + 2] = q.z; v[c + 3] = q.w;
        }
      }
    } else {
#pragma unroll
      for (int c = 0; c < EH; ++c)
        if (c0 + c < E) v[c] = __ldg(row + c);
    }
#pragma unroll
    for (int c = 0; c < EH; ++c) {
      bad = bad || !isfinite(v[c]) && c0 + c < E;
      v[c] = route_key(v[c]);
    }
  }
  bad = bad || __shfl_xor_sync(0xffffffffu, bad ? 1 : 0, 1) != 0;
  // this lane's k largest, in order
  uint32_t taken[EH / 32];
#pragma unroll
  for (int w = 0; w < EH / 32; ++w) taken[w] = 0u;
  float lk[KM];
  int li[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    lk[j] = -CUDART_INF_F;
    li[j] = c0;
    if (j < k) {
      float best = 0.0f;
      int bi = -1;
#pragma unroll
      for (int c = 0; c < EH; ++c) {
        const bool free = ((taken[c >> 5] >> (c & 31)) & 1u) == 0u;
        if (free && (bi < 0 || v[c] > best)) {   // strict: the lower id keeps a tie
          best = v[c];
          bi = c;
        }
      }
#pragma unroll
      for (int w = 0; w < EH / 32; ++w)
        if ((bi >> 5) == w) taken[w] |= 1u << (bi & 31);
      lk[j] = best;
      li[j] = c0 + bi;
    }
  }
  // merge: both lanes step through the two lists in the same way
  const int lane = tid & 31;
  int sel[KM];
  float ex[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) ex[j] = 0.0f;
  float lmax = 0.0f;
  int pa = 0, pb = 0;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    sel[j] = 0;
    if (j < k) {
      const int pm = h ? pb : pa;          // this lane's next entry (< k: 2k entries, k taken)
      float hk = lk[0];
      int hi = li[0];
#pragma unroll
      for (int q = 1; q < KM; ++q)
        if (q == pm) { hk = lk[q]; hi = li[q]; }
      const float ak = __shfl_sync(0xffffffffu, hk, lane & ~1);
      const int ai = __shfl_sync(0xffffffffu, hi, lane & ~1);
      const float bk = __shfl_sync(0xffffffffu, hk, lane | 1);
      const int bidx = __shfl_sync(0xffffffffu, hi, lane | 1);
      const bool take_b = bk > ak;
      const float best = take_b ? bk : ak;
      sel[j] = take_b ? bidx : ai;
      pa += take_b ? 0 : 1;
      pb += take_b ? 1 : 0;
      if (j == 0) lmax = best;
      ex[j] = expf(best - lmax);
    }
  }
  if (valid && h == 0) {
    const float sum = gate_sum8(ex);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k) {
        topk_idx[t * k + j] = sel[j];
        gates[t * k + j] = bad ? 0.0f : ex[j] / sum;
      }
    }
    if (bad) raise_error(err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();   // masks cleared
  if (valid && h == 0) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) atomicOr(&s_mask[4 * sel[j] + (tl >> 5)], 1u << (tl & 31));
  }
  __syncthreads();
  if (valid && h == 0) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) local_rank[t * k + j] = mask_rank(s_mask, sel[j], tl);
  }
  write_block_hist(s_mask, E, block_hist, tid, kTopk2Threads);
}

// (b) E > 128, k <= 8: four threads per token; thread q keeps the k largest of
// columns [q cw, (q + 1) cw) while it reads them, and the four lists are merged
// through lane shuffles in the same total order.
constexpr int kTopk4Threads = 4 * kTpb;

template <int KM>
MOE_DEV void topk_insert(float* tv, int* tix, int k, float kv, int ki) {
  int pos = 0;   // kept entries that stay ahead of the new one
#pragma unroll
  for (int j = 0; j < KM; ++j) pos += (j < k && tix[j] >= 0 && topk_ahead(tv[j], tix[j], kv, ki)) ? 1 : 0;
#pragma unroll
  for (int j = KM - 1; j >= 0; --j) {
    if (j < k && j > pos) {
      tv[j] = tv[j - 1];
      tix[j] = tix[j - 1];
    }
    if (j < k && j == pos) {
      tv[j] = kv;
      tix[j] = ki;
    }
  }
}

template <int KM>
__global__ void __launch_bounds__(kTopk4Threads) route_topk4_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ uint32_t s_mask[256 * 4];
  const int tid = threadIdx.x;
  const int tl = tid >> 2, q = tid & 3;
  const int64_t t = (int64_t)blockIdx.x * kTpb + tl;
  const bool valid = t < T;
  for (int i = tid; i < 4 * E; i += kTopk4Threads) s_mask[i] = 0u;
  float tv[KM];
  int tix[KM];
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    tv[j] = 0.0f;
    tix[j] = -1;
  }
  bool bad = false;
  if (valid) {
    const int cw = (E + 3) >> 2;
    const int c0 = q * cw, c1 = min(E, c0 + cw);
    const float* row = logits + t * E;
#pragma unroll 4
    for (int c = c0; c < c1; ++c) {
      const float x = __ldg(row + c);
      bad = bad || !isfinite(x);
      topk_insert<KM>(tv, tix, k, route_key(x), c);
    }
  }
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {   // every lane ends with the same list
    float ov[KM];
    int oi[KM];
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      ov[j] = __shfl_xor_sync(0xffffffffu, tv[j], off);
      oi[j] = __shfl_xor_sync(0xffffffffu, tix[j], off);
    }
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (oi[j] >= 0) topk_insert<KM>(tv, tix, k, ov[j], oi[j]);
  }
  {   // non-finite logits of the token: OR over its four lanes
    int b = bad ? 1 : 0;
    b |= __shfl_xor_sync(0xffffffffu, b, 1);
    b |= __shfl_xor_sync(0xffffffffu, b, 2);
    bad = b != 0;
  }
  if (valid) {
    float ex[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ex[j] = (j < k && j < KM) ? expf(tv[j < KM ? j : 0] - tv[0]) : 0.0f;
    const float sum = gate_sum8(ex);
#pragma unroll
    for (int j = 0; j < KM; ++j) {
      if (j < k && (j & 3) == q) {
        topk_idx[t * k + j] = tix[j];
        gates[t * k + j] = bad ? 0.0f : ex[j] / sum;
      }
    }
    if (bad && q == 0) raise_error(err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();
  if (valid) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k && (j & 3) == q) atomicOr(&s_mask[4 * tix[j] + (tl >> 5)], 1u << (tl & 31));
  }
  __syncthreads();
  if (valid) {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k && (j & 3) == q) local_rank[t * k + j] = mask_rank(s_mask, tix[j], tl);
  }
  write_block_hist(s_mask, E, block_hist, tid, kTopk4Threads);
}

// (c) any k (used for k > 8): a warp per token, warp-shuffle arg-max rounds;
// eight warps take the block's 128 tokens 16 each.
constexpr int kTopkThreads = 256;

template <int EPL>
__global__ void __launch_bounds__(kTopkThreads) route_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, int32_t* __restrict__ local_rank, int32_t* __restrict__ block_hist,
    int32_t* __restrict__ err) {
  pdl_begin();
  __shared__ int32_t s_sel[kTpb * 32];   // expert of each route of the block
  __shared__ uint32_t s_mask[256 * 4];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kTpb;
  const int ntok = min(kTpb, T - t0);
  for (int i = threadIdx.x; i < 4 * E; i += kTopkThreads) s_mask[i] = 0u;

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
      atomicOr(&s_mask[4 * my_id + (tl >> 5)], 1u << (tl & 31));
    }
    if (token_bad && lane == 0) raise_error(err, MOE_DEVERR_NONFINITE_LOGIT);
  }
  __syncthreads();
  for (int r = threadIdx.x; r < ntok * k; r += kTopkThreads)
    local_rank[(size_t)t0 * k + r] = mask_rank(s_mask, s_sel[r], r / k);
  write_block_hist(s_mask, E, block_hist, threadIdx.x, kTopkThreads);
}

// ---------------------------------------------------------------- scan, slots
// One block of 1024 threads.  Thread (p, e) = (tid / Epad, tid % Epad) owns
// expert e and the p-th contiguous chunk of the routing blocks.  block_hist[b][e]
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
  if (e < E) {
#pragma unroll 8
    for (int b = b0; b < b1; ++b) sum += block_hist[(size_t)b * E + e];
  }
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

// One thread per route (slot = its block's first row for its expert + its rank),
// then one per padding row of each expert's last tile (route_of_slot = -1).
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
    const int b = t / kTpb;
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

}  // namespace

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                              float* gates, int32_t* local_rank, int32_t* block_hist,
                              int32_t* err, cudaStream_t s) {
  const int nb = (T + kTpb - 1) / kTpb;
  if (k <= 8 && E <= 128) {
#define MOE_TOPK_REG(EM, KM)                                                                   \
  launch_pdl(route_topk_reg_kernel<EM, KM>, dim3(nb), dim3(kTpb), 0, s, logits, T, E, k,     \
             topk_idx, gates, local_rank, block_hist, err)
#define MOE_TOPK2(EH, KM)                                                                      \
  launch_pdl(route_topk2_kernel<EH, KM>, dim3(nb), dim3(kTopk2Threads), 0, s, logits, T, E, k, \
             topk_idx, gates, local_rank, block_hist, err)
    if (E <= 32) {
      if (k <= 4) MOE_TOPK_REG(32, 4); else MOE_TOPK_REG(32, 8);
    } else if (E <= 64) {
      if (k <= 4) MOE_TOPK2(32, 4); else MOE_TOPK2(32, 8);
    } else {
      if (k <= 4) MOE_TOPK2(64, 4); else MOE_TOPK2(64, 8);
    }
#undef MOE_TOPK2
#undef MOE_TOPK_REG
    return cudaGetLastError();
  }
  if (k <= 8) {
    if (k <= 4)
      launch_pdl(route_topk4_kernel<4>, dim3(nb), dim3(kTopk4Threads), 0, s, logits, T, E, k,
                 topk_idx, gates, local_rank, block_hist, err);
    else
      launch_pdl(route_topk4_kernel<8>, dim3(nb), dim3(kTopk4Threads), 0, s, logits, T, E, k,
                 topk_idx, gates, local_rank, block_hist, err);
    return cudaGetLastError();
  }
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    launch_pdl(route_topk_kernel<1>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx,
               gates, local_rank, block_hist, err);
  else if (epl <= 2)
    launch_pdl(route_topk_kernel<2>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx,
               gates, local_rank, block_hist, err);
  else if (epl <= 4)
    launch_pdl(route_topk_kernel<4>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx,
               gates, local_rank, block_hist, err);
  else
    launch_pdl(route_topk_kernel<8>, dim3(nb), dim3(kTopkThreads), 0, s, logits, T, E, k, topk_idx,
               gates, local_rank, block_hist, err);
  return cudaGetLastError();
}

cudaError_t launch_route_scan(int32_t* block_hist, int n_blocks, int E, int32_t* counts,
                              int32_t* offsets, int32_t* tile_offsets, cudaStream_t s) {
  int e_pad = 4;
  while (e_pad < E) e_pad <<= 1;   // E <= 256 -> at least 4 chunks per expert
  launch_pdl(route_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, block_hist, n_blocks, E, e_pad,
             counts, offsets, tile_offsets);
  return cudaGetLastError();
}

cudaError_t launch_route_slots(const int32_t* topk_idx, const int32_t* local_rank,
                               const int32_t* block_base, const int32_t* counts,
                               const int32_t* tile_offsets, int T, int E, int k, int64_t rows_max,
                               int32_t* slot_of_route, int32_t* route_of_slot, int32_t* err,
                               cudaStream_t s) {
  const int64_t n = (int64_t)T * k + (int64_t)E * kTileM;
  const int nb = (int)((n + 255) / 256);
  launch_pdl(route_slots_kernel, dim3(nb), dim3(256), 0, s, topk_idx, local_rank, block_base,
             counts, tile_offsets, T, E, k, rows_max, slot_of_route, route_of_slot, err);
  return cudaGetLastError();
}

cudaError_t launch_route(int T, int d, int E, int k, int64_t rows_max, const void* x,
                         const void* w_router, const float* bias, float* logits,
                         int32_t* topk_idx, float* gates, int32_t* counts, int32_t* offsets,
                         int32_t* tile_offsets, int32_t* slot_of_route, int32_t* route_of_slot,
                         int32_t* err, int32_t* hist, int32_t* rank, cudaStream_t s) {
  cudaError_t e;
  if (w_router != nullptr) {
    GemmLaunch g = {};
    g.op = OP_ROUTER;
    g.T = T; g.d = d; g.E = E; g.f = 128;
    g.rows_max = rows_max;
    g.a0 = x; g.w0 = w_router; g.bias = bias; g.out0 = logits; g.err = err;
    if ((e = launch_grouped_gemm(g, s)) != cudaSuccess) return e;
  }
  if ((e = launch_route_topk(logits, T, E, k, topk_idx, gates, rank, hist, err, s)) != cudaSuccess)
    return e;
  const int nb = (T + kTpb - 1) / kTpb;
  if ((e = launch_route_scan(hist, nb, E, counts, offsets, tile_offsets, s)) != cudaSuccess) return e;
  return launch_route_slots(topk_idx, rank, hist, counts, tile_offsets, T, E, k, rows_max,
                            slot_of_route, route_of_slot, err, s);
}

MOE_CHECK_WORD_ACCESSOR(route)

}  // namespace moe
