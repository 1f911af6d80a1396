// MXFP8 kernels (sm_103a): E4M3 values with one E8M0 scale per 32 values along
// the contraction axis ("Supercharging Olmo-core for Efficient and Scalable MoE
// Training", Abstract and Section 24 Evidence 10: MXFP8 with shared block
// scales, 33/32 byte per value; Section 24.3: the quantiser emits a layout the
// GEMM consumes without a conversion pass).
//   quantize_rows   K along the row: codes keep the orientation
//   quantize_cols   K along the column: codes are written transposed (K-major),
//                   the second weight cache of the data-gradient GEMMs
//   dispatch_mxfp8  x[t] quantised once, then written to its k expert rows
//   dequantize      codes + scales -> bf16 (the global dequantisation that
//                   feeds the BF16 weight-gradient GEMMs, Section 24 Evidence 7)
// Scales are stored at sf_offset() (common.cuh), the layout the GEMM copies
// into tensor memory.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// One thread per 32-value block of a [rows, cols] bf16 matrix (K = cols).
// Output row of input row r: r, or with `group` > 0 (interleaving two matrices
// into one of 2*rows rows): (r / group) * 2 * group + offset + r % group.
// `group` is a power of two (the launchers refuse others).
MOE_DEV int64_t interleaved_row(int64_t r, int group, int offset) {
  if (group <= 0) return r;
  const int sh = __ffs(group) - 1;
  return ((r >> sh) << (sh + 1)) + offset + (r & (group - 1));
}
__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(
    const uint4* __restrict__ src, int64_t nblocks, int rows, int cols, int group, int offset,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  pdl_begin();
  const int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x;
  if (i >= nblocks) return;
  const int kb = cols / 32;
  const int64_t per_mat = (int64_t)rows * kb;
  const int64_t mat = i / per_mat;
  const int64_t rem = i - mat * per_mat;
  const int64_t r = rem / kb;
  const int b = (int)(rem - r * kb);
  const int64_t out_rows = group > 0 ? 2 * (int64_t)rows : rows;
  const int64_t ro = interleaved_row(r, group, offset);
  float v[32];
#pragma unroll
  for (int u = 0; u < 4; ++u) unpack8(__ldg(src + i * 4 + u), v + 8 * u);
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int s = mx_scale_exp(amax);
  const float inv = exp2i(-s);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] *= inv;
  uint2* out = reinterpret_cast<uint2*>(q + ((size_t)mat * out_rows + ro) * cols + (size_t)b * 32);
#pragma unroll
  for (int u = 0; u < 4; ++u) out[u] = e4m3x8(v + 8 * u);
  sf[(size_t)mat * out_rows * kb + sf_offset(ro, b, kb)] = (uint8_t)(s + 127);
}

// K along the column: src [K=rows, N=cols] bf16 -> q [N, K] (K-major) with
// scales of the [N, K] operand.  Tile: 128 K x 64 N per block.
constexpr int kTK = 128, kTN = 64;
__global__ void __launch_bounds__(kQThreads) quantize_cols_kernel(
    const __nv_bfloat16* __restrict__ src, int K, int N, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sf) {
  pdl_begin();
  __shared__ __nv_bfloat16 tile[kTK][kTN];
  const int mat = blockIdx.z;
  const int k0 = blockIdx.y * kTK;
  const int n0 = blockIdx.x * kTN;
  const __nv_bfloat16* s = src + (size_t)mat * K * N;
  // 128 rows x 128 bytes: 1024 16-byte vectors, 4 per thread
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int idx = threadIdx.x + u * kQThreads;
    const int row = idx >> 3, col = (idx & 7) * 8;
    *reinterpret_cast<uint4*>(&tile[row][col]) =
        __ldg(reinterpret_cast<const uint4*>(s + (size_t)(k0 + row) * N + n0 + col));
  }
  __syncthreads();
  const int n = threadIdx.x & 63;
  const int kb = threadIdx.x >> 6;          // 4 blocks of 32 along K
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = __bfloat162float(tile[kb * 32 + j][n]);
    amax = fmaxf(amax, fabsf(v[j]));
  }
  const int e = mx_scale_exp(amax);
  const float inv = exp2i(-e);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] *= inv;
  const size_t row_out = (size_t)n0 + n;
  uint2* out = reinterpret_cast<uint2*>(q + (size_t)mat * N * K + row_out * K + k0 + kb * 32);
#pragma unroll
  for (int u = 0; u < 4; ++u) out[u] = e4m3x8(v + 8 * u);
  sf[(size_t)mat * N * (K / 32) + sf_offset((int64_t)row_out, (k0 / 32) + kb, K / 32)] =
      (uint8_t)(e + 127);
}

// Both orientations of a weight from one read: src [R, C] bf16 per matrix ->
// (1) q_r [R, C] blocked along C (rows interleaved by `group`/`offset` as in
// quantize_rows_kernel) and (2) q_c [C, R] blocked along R (the transpose, as
// in quantize_cols_kernel).  Tile: 128 rows x 128 columns (32 KB) staged in
// shared memory from eight 16-byte loads in flight per thread, 16-byte chunk c
// of row r at chunk c ^ (r % 16), which keeps the row reads of (1) and the
// column reads of (2) free of bank conflicts.  (1): a thread quantises two
// 32-value blocks of one row.  (2): a thread quantises one 32-row block of two
// adjacent columns (32-bit reads).  Both code sets are then staged in the
// tile's memory (16 KB each) and stored as whole 128-byte rows.
constexpr int kBR = 128, kBC = 128;
__global__ void __launch_bounds__(kQThreads, 4) quantize_both_kernel(
    const __nv_bfloat16* __restrict__ src, int R, int C, int group, int offset,
    uint8_t* __restrict__ q_r, uint8_t* __restrict__ s_r, uint8_t* __restrict__ q_c,
    uint8_t* __restrict__ s_c) {
  pdl_begin();
  __shared__ __align__(16) uint8_t tile[kBR * kBC * 2];
  const int mat = blockIdx.z;
  const int k0 = blockIdx.y * kBR;
  const int n0 = blockIdx.x * kBC;
  const __nv_bfloat16* sm = src + (size_t)mat * R * C;
  const int64_t out_rows = group > 0 ? 2 * (int64_t)R : R;
  const int cb = C / 32;
  constexpr int kLoads = kBR * kBC / 8 / kQThreads;   // 8
  uint4 raw[kLoads];   // all loads in flight before any is used
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int idx = threadIdx.x + u * kQThreads;
    raw[u] = __ldg(reinterpret_cast<const uint4*>(sm + (size_t)(k0 + (idx >> 4)) * C + n0 +
                                                   (idx & 15) * 8));
  }
#pragma unroll
  for (int u = 0; u < kLoads; ++u) {
    const int idx = threadIdx.x + u * kQThreads;
    const int row = idx >> 4, c = idx & 15;
    *reinterpret_cast<uint4*>(tile + row * 256 + ((c ^ (row & 15)) << 4)) = raw[u];
  }
  __syncthreads();
  // (1) row `rr`, 32-value blocks b0 and b0 + 1 of the tile's four
  const int rr = threadIdx.x >> 1;
  const int b0 = 2 * (threadIdx.x & 1);
  uint4 rcode[4];
  uint32_t rsb = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int b = b0 + h;
    uint32_t pk[16];   // the block's 32 bf16 values, two per word (unpacked at use)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 c4 =
          *reinterpret_cast<const uint4*>(tile + rr * 256 + (((4 * b + u) ^ (rr & 15)) << 4));
      pk[4 * u] = c4.x; pk[4 * u + 1] = c4.y; pk[4 * u + 2] = c4.z; pk[4 * u + 3] = c4.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(pk[j] << 16)),
                               fabsf(__uint_as_float(pk[j] & 0xFFFF0000u))));
    const int sx = mx_scale_exp(amax);
    const float inv = exp2i(-sx);
    uint2 q[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        t[2 * i] = __uint_as_float(pk[4 * g + i] << 16) * inv;
        t[2 * i + 1] = __uint_as_float(pk[4 * g + i] & 0xFFFF0000u) * inv;
      }
      q[g] = e4m3x8(t);
    }
    rcode[2 * h] = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
    rcode[2 * h + 1] = make_uint4(q[2].x, q[2].y, q[3].x, q[3].y);
    rsb |= (uint32_t)(sx + 127) << (8 * h);
  }
  {   // blocks b0 and b0 + 1 (b0 even): adjacent scale bytes
    const int64_t ro = interleaved_row(k0 + rr, group, offset);
    *reinterpret_cast<uint16_t*>(s_r + (size_t)mat * out_rows * cb +
                                 sf_offset(ro, n0 / 32 + b0, cb)) = (uint16_t)rsb;
  }
  // (2) columns 2 cp and 2 cp + 1, rows 32 kb .. 32 kb + 31
  const int cpair = threadIdx.x & 63;
  const int kb = threadIdx.x >> 6;
  uint32_t w[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int r = 32 * kb + j;
    w[j] = *reinterpret_cast<const uint32_t*>(tile + r * 256 + (((cpair >> 2) ^ (r & 15)) << 4) +
                                              4 * (cpair & 3));
  }
  uint4 ccode[4];
#pragma unroll
  for (int i = 0; i < 2; ++i) {   // column 2 cpair + i: the low (i = 0) or high bf16 halves
    auto val = [&](int j) {
      return __uint_as_float(i ? (w[j] & 0xFFFF0000u) : (w[j] << 16));
    };
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(val(j)));
    const int e = mx_scale_exp(amax);
    const float inv = exp2i(-e);
    uint2 q[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float t[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) t[j] = val(8 * g + j) * inv;
      q[g] = e4m3x8(t);
    }
    ccode[2 * i] = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
    ccode[2 * i + 1] = make_uint4(q[2].x, q[2].y, q[3].x, q[3].y);
    s_c[(size_t)mat * C * (R / 32) + sf_offset((int64_t)n0 + 2 * cpair + i, (k0 / 32) + kb, R / 32)] =
        (uint8_t)(e + 127);
  }
  // Stage both code sets in the tile's memory once every read of it is done:
  // q_r codes of tile row r in bytes [0, 16 KB), 16-byte chunk c at c ^ (r % 8);
  // q_c codes of output row n in [16 KB, 32 KB), chunk c at c ^ ((n / 2) % 8).
  __syncthreads();
  uint8_t* st_r = tile;
  uint8_t* st_c = tile + kBR * kBC;
#pragma unroll
  for (int q = 0; q < 4; ++q)   // chunks 2 b0 .. 2 b0 + 3 of row rr
    *reinterpret_cast<uint4*>(st_r + rr * 128 + (((2 * b0 + q) ^ (rr & 7)) << 4)) = rcode[q];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = 2 * cpair + i;
#pragma unroll
    for (int q = 0; q < 2; ++q)   // chunks 2 kb, 2 kb + 1 of output row n
      *reinterpret_cast<uint4*>(st_c + n * 128 + (((2 * kb + q) ^ ((n >> 1) & 7)) << 4)) =
          ccode[2 * i + q];
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int idx = threadIdx.x + u * kQThreads;   // 1024 16-byte pieces per code set
    const int rn = idx >> 3, c = idx & 7;
    const int64_t ro = interleaved_row(k0 + rn, group, offset);
    *reinterpret_cast<uint4*>(q_r + ((size_t)mat * out_rows + ro) * C + n0 + 16 * c) =
        *reinterpret_cast<const uint4*>(st_r + rn * 128 + ((c ^ (rn & 7)) << 4));
    *reinterpret_cast<uint4*>(q_c + (size_t)mat * C * R + ((size_t)n0 + rn) * R + k0 + 16 * c) =
        *reinterpret_cast<const uint4*>(st_c + rn * 128 + ((c ^ ((rn >> 1) & 7)) << 4));
  }
}

// Warp per token: a lane holds 8 values of a 256-column chunk; 4 lanes form a
// 32-value block.  Codes and scales go to all k expert rows; padding rows get
// zero codes and scale byte 127 (2^0).
__global__ void __launch_bounds__(kQThreads) dispatch_mxfp8_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ slot_of_route,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ tile_offsets, int T, int d,
    int E, int k, int token_blocks, uint8_t* __restrict__ xq, uint8_t* __restrict__ xs,
    uint4* __restrict__ xdq) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int warps = kQThreads / 32;
  const int nv = d / 8;
  const int kb = d / 32;
  if (blockIdx.x >= token_blocks) {
    const int p = (blockIdx.x - token_blocks) * warps + (threadIdx.x >> 5);
    if (p >= E * kTileM) return;
    const int e = p / kTileM;
    const int row = tile_offsets[e] * kTileM + counts[e] + (p % kTileM);
    if (row >= tile_offsets[e + 1] * kTileM) return;
    MOE_CHECKED(row, rows_max_of(T, k, E)) {
      uint2* dst = reinterpret_cast<uint2*>(xq + (size_t)row * d);
      for (int c = lane; c < nv; c += 32) dst[c] = make_uint2(0, 0);
      for (int b = lane; b < kb; b += 32) xs[sf_offset(row, b, kb)] = 127;
      if (xdq != nullptr)
        for (int c = lane; c < nv; c += 32) xdq[(size_t)row * nv + c] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int my_slot = (lane < k) ? slot_of_route[(size_t)t * k + lane] : 0;
  for (int c0 = 0; c0 < nv; c0 += 32) {      // warp-uniform
    const int c = c0 + lane;
    const bool ok = c < nv;
    float v[8];
    if (ok) unpack8(__ldg(x + (size_t)t * nv + c), v);
    else
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int s = mx_scale_exp(amax);
    const float inv = exp2i(-s);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= inv;
    const uint2 codes = e4m3x8(v);
    // dequantised copy (the dequantiser's arithmetic: code value x 2^s, bf16)
    uint4 dq = make_uint4(0, 0, 0, 0);
    if (xdq != nullptr) {
      const float sc = exp2i(s);
      float f[8];
      e4m3x2_to_f32(codes.x & 0xFFFFu, f[0], f[1]);
      e4m3x2_to_f32(codes.x >> 16, f[2], f[3]);
      e4m3x2_to_f32(codes.y & 0xFFFFu, f[4], f[5]);
      e4m3x2_to_f32(codes.y >> 16, f[6], f[7]);
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] *= sc;
      dq = pack8(f);
    }
    for (int j = 0; j < k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);
      if (ok) MOE_CHECKED(slot, rows_max_of(T, k, E)) {
        reinterpret_cast<uint2*>(xq + (size_t)slot * d)[c] = codes;
        if ((lane & 3) == 0) xs[sf_offset(slot, c / 4, kb)] = (uint8_t)(s + 127);
        if (xdq != nullptr) xdq[(size_t)slot * nv + c] = dq;
      }
    }
  }
}

// One thread per 16 codes of a [rows, K] MXFP8 operand -> bf16 [rows, K].
__global__ void __launch_bounds__(kQThreads) dequantize_kernel(
    const uint4* __restrict__ q, const uint8_t* __restrict__ sf, int64_t nvec, int K,
    uint4* __restrict__ out) {
  pdl_begin();
  const int64_t i = (int64_t)blockIdx.x * kQThreads + threadIdx.x;
  if (i >= nvec) return;
  const int per_row = K / 16;
  const int64_t r = i / per_row;
  const int c16 = (int)(i - r * per_row);
  const int b = c16 / 2;
  const float scale = exp2i((int)sf[sf_offset(r, b, K / 32)] - 127);
  const uint4 v = __ldg(q + i);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[16];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    e4m3x2_to_f32(w[u] & 0xFFFFu, f[4 * u + 0], f[4 * u + 1]);
    e4m3x2_to_f32(w[u] >> 16, f[4 * u + 2], f[4 * u + 3]);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) f[j] *= scale;
  out[2 * i] = pack8(f);
  out[2 * i + 1] = pack8(f + 8);
}

}  // namespace

cudaError_t launch_quantize_mxfp8(int batch, int rows, int cols, int block_axis, const void* src,
                                  uint8_t* q, uint8_t* sf, cudaStream_t s, int group, int offset) {
  if (group < 0 || (group & (group - 1)) != 0) return cudaErrorInvalidValue;
  if (block_axis == 1) {
    const int64_t n = (int64_t)batch * rows * (cols / 32);
    launch_pdl(quantize_rows_kernel, dim3((unsigned)((n + kQThreads - 1) / kQThreads)), dim3(kQThreads), 0, s, 
        static_cast<const uint4*>(src), n, rows, cols, group, offset, q, sf);
  } else {
    dim3 grid((unsigned)(cols / kTN), (unsigned)(rows / kTK), (unsigned)batch);
    launch_pdl(quantize_cols_kernel, dim3(grid), dim3(kQThreads), 0, s, static_cast<const __nv_bfloat16*>(src), rows,
                                                    cols, q, sf);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8_both(int batch, int rows, int cols, const void* src, int group,
                                       int offset, uint8_t* q_rows, uint8_t* sf_rows,
                                       uint8_t* q_cols, uint8_t* sf_cols, cudaStream_t s) {
  if (group < 0 || (group & (group - 1)) != 0) return cudaErrorInvalidValue;
  dim3 grid((unsigned)(cols / kBC), (unsigned)(rows / kBR), (unsigned)batch);
  launch_pdl(quantize_both_kernel, grid, dim3(kQThreads), 0, s,
             static_cast<const __nv_bfloat16*>(src), rows, cols, group, offset, q_rows, sf_rows,
             q_cols, sf_cols);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_mxfp8(const void* x, const int32_t* slot_of_route,
                                  const int32_t* counts, const int32_t* tile_offsets, int T, int d,
                                  int E, int k, uint8_t* xq, uint8_t* xs, cudaStream_t s,
                                  void* xdq) {
  const int warps = kQThreads / 32;
  const int tb = (T + warps - 1) / warps;
  const int pb = (E * kTileM + warps - 1) / warps;
  launch_pdl(dispatch_mxfp8_kernel, dim3(tb + pb), dim3(kQThreads), 0, s, static_cast<const uint4*>(x), slot_of_route,
                                                      counts, tile_offsets, T, d, E, k, tb, xq, xs,
                                                      static_cast<uint4*>(xdq));
  return cudaGetLastError();
}

cudaError_t launch_dequantize_mxfp8(const uint8_t* q, const uint8_t* sf, int64_t rows, int K,
                                    void* out, cudaStream_t s) {
  const int64_t nvec = rows * (K / 16);
  launch_pdl(dequantize_kernel, dim3((unsigned)((nvec + kQThreads - 1) / kQThreads)), dim3(kQThreads), 0, s, 
      reinterpret_cast<const uint4*>(q), sf, nvec, K, static_cast<uint4*>(out));
  return cudaGetLastError();
}

MOE_CHECK_WORD_ACCESSOR(quant)

}  // namespace moe
