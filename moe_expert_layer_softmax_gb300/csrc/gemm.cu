// Device-scheduled grouped GEMM on tcgen05 tensor cores (sm_103a).
//
// "Supercharging Olmo-core for Efficient and Scalable MoE Training", Abstract:
// the expert GEMMs are grouped GEMMs scheduled on the device from routing
// metadata that never leaves the GPU; the article "Olmo-core 3: an open training
// stack for trillion-parameter MoE" (section "Olmo-core 3's answer: experts
// resident, data routed") adds that
// they run the uneven per-expert shapes without padding to a common capacity.
// Here each expert's rows are padded only to the 128-row tile, and the tile
// schedule is read from the device-resident tile_offsets.
//
// Kernel structure (persistent, one CTA per SM, 320 threads):
//   warp 0     TMA producer: 128-byte-swizzled A/B tiles into a 192 KB ring
//              (6 stages of 32 KB on CTA pairs, 4 of 48 KB on single CTAs,
//              up to 12 for the narrow router tile, 5 of 33 KB for MXFP8)
//   warp 1     TMEM allocator and single-thread tcgen05.mma issuer (bf16 or
//              block-scaled fp8 in, fp32 accumulators in tensor memory, two
//              accumulators so the epilogue of one tile overlaps the main loop
//              of the next)
//   warps 2-9  epilogue, two warps per TMEM lane quarter (each takes half of
//              the tile's columns): tcgen05.ld -> fused SwiGLU /
//              SwiGLU-backward / fp32 / router math -> swizzled shared-memory
//              staging -> TMA bulk stores (direct stores for the router and
//              the MXFP8 epilogues)
// CTA pairs (clusters of 2, the bf16 data GEMMs): one 256-row tile per pair
// with tcgen05.mma.cta_group::2; each CTA stages its 128 A rows and half of B,
// the even CTA issues the MMAs (see "CTA pairs" below).
// Weight gradients on the natural MXFP8 layout (the third template flag): B
// arrives as E4M3 codes + scale atoms and 8 more warps (converters) write the
// dequantised bf16 B tile for each stage; 576 threads.
// Every wait is bounded (error word + abort flag); an aborted CTA waits for
// its own copies in flight and frees its tensor memory before returning.
//
// Schedules:
//   DENSE   (router)       tiles = ceil(T/128) x n_tiles (x 2 K halves when the
//                          row tiles fill at most half the SMs), K = d
//   MGROUP  (fwd / dgrad)  tiles = tile_offsets[E] x n_tiles; a tile's expert is
//                          found by binary search in tile_offsets
//   KGROUP  (wgrad)        tiles = E x (M/128) x n_tiles, the K loop runs over
//                          the expert's (padded, zero-filled) rows
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

enum Mode { MODE_DENSE = 0, MODE_MGROUP = 1, MODE_KGROUP = 2 };
enum Epi {
  EPI_BF16 = 0, EPI_SWIGLU_FWD = 1, EPI_SWIGLU_BWD = 2, EPI_F32 = 3, EPI_ROUTER = 4,
  EPI_SWIGLU_FWD_MX = 5,  // H, U bf16 + A quantised to MXFP8 (one block per 32 columns)
  EPI_SWIGLU_BWD_MX = 6,  // dH, dU bf16 + both quantised to MXFP8
};

constexpr int kMaxStages = 12;
constexpr int kRingBytes = 192 * 1024;
constexpr int kStageOutBytes = 16 * 1024;     // per column half: 128 rows x 128 bytes
constexpr int kBK = 64;                       // bf16 elements of K per stage (128 bytes)
constexpr int kABytes = kTileM * kBK * 2;     // 16 KB
constexpr int kBBytesMax = 256 * kBK * 2;     // 32 KB
constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kMaxE = 256;
constexpr uint32_t kTmemCols = 512;           // two 256-column fp32 accumulators

// Weight gradients whose B operand stays in the forward's MXFP8 layout (codes
// with one E8M0 scale per 32 columns of a row) and is dequantised inside the
// kernel: each ring stage holds the TMA-loaded A tile, 64 rows x 128 codes of
// B and the 512-byte scale atom covering them; converter warps write the bf16
// B tile into one of kDqSlots slots after the stages, in the 128-byte-swizzled
// M/N-major layout a TMA load of the dequantised tensor would have produced.
constexpr int kConvWarps = 8;
constexpr int kThreadsDq = kThreads + 32 * kConvWarps;
constexpr int kDqRawBytes = kBK * 128;                // 64 rows x 128 E4M3 codes
constexpr int kDqStageBytes = 25 * 1024;              // A + codes + scale atom, 1 KB multiple
constexpr int kDqSlotBytes = kBK * 128 * 2;           // one bf16 B tile (64 x 128)
constexpr int kDqSlots = 4;
constexpr int kDqStages = (kRingBytes - kDqSlots * kDqSlotBytes) / kDqStageBytes;
static_assert(kABytes + kDqRawBytes + 512 <= kDqStageBytes, "stage layout");
static_assert(kDqStages >= 4 && kDqStages <= kMaxStages, "ring depth");
static_assert(kDqSlots >= 2 && kDqSlots <= 4, "B slots");

struct __align__(8) Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t fin;
  uint64_t rawfull[kMaxStages];  // in-kernel dequantisation: this CTA's codes + scales landed
  uint64_t bfull[4];             // converted B slot ready (even CTA, both CTAs' converters)
  uint64_t bempty[4];            // B slot free again (the pair's MMAs that read it are done)
  uint64_t hufull[2];            // MXFP8 SwiGLU backward, per column half: H and U chunk landed,
  uint64_t huwritten[2];         //   dH and dU written over it by the half's 128 epilogue threads,
  uint64_t codefree[2];          //   the half's code buffer read by the previous chunk's stores
  uint32_t tmem_base;
  int abort;
  int32_t tile_off[kMaxE + 1];
  int32_t pair_off[kMaxE + 1];   // CTA pairs, M-grouped: exclusive scan of ceil(m-tiles / 2)
                                 // per expert; K-grouped: the experts in tile order
};

// the dynamic shared memory is declared 1024-byte aligned (the swizzled tiles
// need it), so no alignment slack is requested
constexpr int kSmemBytes = kRingBytes + 2 * kStageOutBytes + (int)sizeof(Ctl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct Params {
  int mode;
  int epi;
  int a_mn, b_mn;        // operand major-ness (1 = M/N-major, 0 = K-major)
  int b_dual;            // B tile = 128 rows of map B0 + 128 rows of map B1 (K-major)
  int E;
  const int32_t* tile_offsets;
  int m_tiles;           // DENSE: M tiles; KGROUP: M/128 per expert
  int m_valid;           // DENSE: valid rows (T)
  int n_tiles;
  int BN;                // MMA N (256 when b_dual)
  int n_valid;           // ROUTER: valid columns (E)
  int n_cols;            // bf16 pairs with N = 128 (mod 256): N; the last 256-wide tile's
                         // second half lies past it (0: every tile column is valid)
  int k_steps;           // DENSE/MGROUP: K / 64
  int k_parts;           // DENSE: K split into this many parts (1 or 2), summed atomically
  int k_split;           // DENSE/MGROUP: steps >= k_split read maps A1/B1
  int m_split;           // KGROUP: M tiles >= m_split read A1 and write out1
  int b_group_rows;      // expert stride in the rows of B's 2-D view
  int stages;            // ring depth
  int stage_bytes;       // stage stride in the ring, a multiple of 1024
  int tx_bytes;          // bytes the producer's copies deliver per stage
  int kstep;             // K elements per stage: 64 bf16 or 128 fp8 (128 bytes either way)
  int acc_cols;          // TMEM columns per accumulator (256, or 128 for MXFP8 tiles)
  // MXFP8 operands: scales in the sf_offset layout, sf_k* = K / 128 atoms per row block
  const uint8_t* sfa0;
  const uint8_t* sfa1;
  const uint8_t* sfb0;
  const uint8_t* sfb1;
  int sf_ka, sf_kb;
  void* out3;
  uint8_t* osf0;         // scales of quantised outputs (sf_offset layout, osf_kb blocks/row)
  uint8_t* osf1;
  int osf_kb;
  int inject_stall;      // test hook: the producer issues nothing (see moe_debug_inject_stall)
  int tma_store;         // epilogue writes through swizzled smem + TMA bulk stores
  int64_t out_rows_per_group;  // KGROUP TMA store: rows of one expert's output (M)
  int num_acc;           // TMEM accumulators (2: the epilogue overlaps the next tile)
  int tmem_cols;         // TMEM columns allocated
  int pair_half_bytes;   // CTA pairs: bytes one CTA's copies deliver per stage
  int dq_b;              // B is MXFP8 codes (map B0, uint8) dequantised in the kernel
  const uint8_t* sfq;    //   its scales (sf_offset layout)
  int sfq_k;             //   scale atoms per 128-row block (B columns / 128)
  void* out0;
  void* out1;
  void* out2;
  const void* aux0;
  const void* aux1;
  const float* bias;
  int64_t rows_max;      // rows of the dispatched row buffers
  int64_t ldo;           // leading dimension (elements) of outputs and aux
  int64_t out_group_stride;  // KGROUP: elements between experts' outputs
  int32_t* err;
};

struct TileInfo {
  int e, m_tile, n_tile, k0row, ks;
  int kb;   // DENSE split-K: first K step of this part
};

MOE_DEV int find_group(const int32_t* off, int E, int m_tile) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= m_tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

MOE_DEV int total_tiles(const Params& p, const int32_t* off) {
  if (p.mode == MODE_DENSE) return p.m_tiles * p.n_tiles * p.k_parts;
  if (p.mode == MODE_MGROUP) return off[p.E] * p.n_tiles;
  return p.E * p.m_tiles * p.n_tiles;
}

MOE_DEV TileInfo decode_tile(const Params& p, const int32_t* off, int t) {
  TileInfo ti;
  ti.kb = 0;
  if (p.mode == MODE_DENSE) {
    const int part = t % p.k_parts;
    const int mt = t / p.k_parts;
    ti.m_tile = mt / p.n_tiles;
    ti.n_tile = mt - ti.m_tile * p.n_tiles;
    ti.e = 0;
    ti.k0row = 0;
    ti.ks = p.k_steps / p.k_parts;
    ti.kb = part * ti.ks;
    return ti;
  }
  if (p.mode == MODE_KGROUP) {
    const int per = p.m_tiles * p.n_tiles;
    ti.e = t / per;
    const int r = t - ti.e * per;
    ti.m_tile = r / p.n_tiles;
    ti.n_tile = r - ti.m_tile * p.n_tiles;
    ti.k0row = off[ti.e] * kTileM;
    ti.ks = (off[ti.e + 1] - off[ti.e]) * (kTileM / kBK);
  } else {
    ti.m_tile = t / p.n_tiles;
    ti.n_tile = t - ti.m_tile * p.n_tiles;
    ti.e = (p.mode == MODE_MGROUP) ? find_group(off, p.E, ti.m_tile) : 0;
    ti.k0row = 0;
    ti.ks = p.k_steps;
  }
  return ti;
}

// logistic sigmoid with the fast reciprocal (the results are stored in bf16)
MOE_DEV float sigmoid_f(float h) { return __fdividef(1.0f, 1.0f + __expf(-h)); }
MOE_DEV float silu_f(float h) { return h * sigmoid_f(h); }

// ------------------------------------------------------------------ roles
// One stage's TMA loads (and, for MXFP8, the stage's scale atoms).
template <bool MX>
MOE_DEV void stage_loads(const Params& p, const TileInfo& ti, int ks, uint8_t* sa, uint64_t* fb,
                         const CUtensorMap* tA0, const CUtensorMap* tA1, const CUtensorMap* tB0,
                         const CUtensorMap* tB1) {
  uint8_t* sb = sa + kABytes;
  if (p.mode == MODE_KGROUP) {
    const bool hi = ti.m_tile >= p.m_split;
    const CUtensorMap* ma = hi ? tA1 : tA0;
    const int mcol = (ti.m_tile - (hi ? p.m_split : 0)) * kTileM;
    const int krow = ti.k0row + ks * kBK;
    tma_load_2d(sa, ma, fb, mcol, krow);
    tma_load_2d(sa + kABytes / 2, ma, fb, mcol + 64, krow);
    for (int i = 0; i < p.BN / 64; ++i)
      tma_load_2d(sb + i * 8192, tB0, fb, ti.n_tile * p.BN + 64 * i, krow);
    return;
  }
  const bool src1 = ks >= p.k_split;
  const int kk = (src1 ? ks - p.k_split : ks) * p.kstep;
  const CUtensorMap* mb = src1 ? tB1 : tB0;
  tma_load_2d(sa, src1 ? tA1 : tA0, fb, kk, ti.m_tile * kTileM);
  if constexpr (MX) {
    // the stage's 128x4 A scales and BNx4 B scales: 512-byte atoms
    uint8_t* sf = sb + p.BN * 128;
    const int brow = ti.e * p.b_group_rows + ti.n_tile * p.BN;
    bulk_load(sf, (src1 ? p.sfa1 : p.sfa0) + ((size_t)ti.m_tile * p.sf_ka + kk / 128) * 512, 512,
              fb);
    for (int i = 0; i < p.BN / 128; ++i)
      bulk_load(sf + 512 * (1 + i),
                (src1 ? p.sfb1 : p.sfb0) + ((size_t)(brow / 128 + i) * p.sf_kb + kk / 128) * 512,
                512, fb);
  }
  if (p.b_mn) {
    const int krow = ti.e * p.b_group_rows + kk;
    for (int i = 0; i < p.BN / 64; ++i)
      tma_load_2d(sb + i * 8192, mb, fb, ti.n_tile * p.BN + 64 * i, krow);
  } else if (p.b_dual) {
    const int row = ti.e * p.b_group_rows + ti.n_tile * 128;
    tma_load_2d(sb, tB0, fb, kk, row);
    tma_load_2d(sb + kBBytesMax / 2, tB1, fb, kk, row);
  } else {
    tma_load_2d(sb, mb, fb, kk, ti.e * p.b_group_rows + ti.n_tile * p.BN);
  }
}

template <bool MX>
MOE_DEV void producer(const Params& p, Ctl& s, uint8_t* ring, const CUtensorMap* tA0,
                      const CUtensorMap* tA1, const CUtensorMap* tB0, const CUtensorMap* tB1) {
  if (p.inject_stall) return;   // the consumers' bounded waits must run out
  const int nt = total_tiles(p, s.tile_off);
  const uint32_t bytes = (uint32_t)p.tx_bytes;
  int stage = 0;
  uint32_t phase = 0;
  long issued = 0;
  bool ok = true;
  for (int t = blockIdx.x; ok && t < nt; t += gridDim.x) {
    const TileInfo ti = decode_tile(p, s.tile_off, t);
    for (int ks = 0; ks < ti.ks; ++ks) {
      if (!mbar_wait(&s.empty[stage], phase ^ 1u, &s.abort, p.err)) { ok = false; break; }
      uint64_t* fb = &s.full[stage];
      uint8_t* sa = ring + stage * p.stage_bytes;
      mbar_arrive_expect_tx(fb, bytes);
      ++issued;
      stage_loads<MX>(p, ti, ti.kb + ks, sa, fb, tA0, tA1, tB0, tB1);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    // Do not leave the CTA with copies in flight: wait (bounded) for the
    // full barriers of the last `stages` issues.  Earlier issues completed
    // before their stage was released for reuse.
    for (long i = (issued > p.stages ? issued - p.stages : 0); i < issued; ++i) {
      const int st = (int)(i % p.stages);
      const uint32_t par = (uint32_t)((i / p.stages) & 1);
      const uint32_t a = smem_u32(&s.full[st]);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(a, par)) {
        if (globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
  }
}

template <bool MX>
MOE_DEV void mma_issuer(const Params& p, Ctl& s, uint8_t* ring, uint32_t tmem_base) {
  const int nt = total_tiles(p, s.tile_off);
  const int n_mma = p.b_dual ? 256 : p.BN;
  const uint32_t idesc = idesc_bf16_f32(kTileM, n_mma, p.a_mn, p.b_mn);
  int stage = 0;
  uint32_t phase = 0;
  int it = 0;
  bool ok = true;
  for (int t = blockIdx.x; ok && t < nt; t += gridDim.x, ++it) {
    const TileInfo ti = decode_tile(p, s.tile_off, t);
    const int acc = it & 1;
    const uint32_t use = (uint32_t)(it >> 1);
    if (!mbar_wait(&s.tempty[acc], (use & 1u) ^ 1u, &s.abort, p.err)) { ok = false; break; }
    tc_fence_after();
    const uint32_t tmem_d = tmem_base + (uint32_t)(acc * p.acc_cols);
    for (int ks = 0; ks < ti.ks; ++ks) {
      if (!mbar_wait(&s.full[stage], phase, &s.abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t a_addr = smem_u32(ring + stage * p.stage_bytes);
      const uint32_t b_addr = a_addr + kABytes;
      if constexpr (MX) {
        // scales of this stage -> tensor memory (columns after both accumulators)
        const uint32_t sf_smem = b_addr + (uint32_t)p.BN * 128u;
        const uint32_t t_sfa = tmem_base + 2u * (uint32_t)p.acc_cols + (uint32_t)stage * 8u;
        const uint32_t t_sfb = t_sfa + 4u;
        tc_cp_32x128b_x4(t_sfa, smem_desc_noswz(sf_smem));
        for (int i = 0; i < p.BN / 128; ++i)
          tc_cp_32x128b_x4(t_sfb + 4u * i, smem_desc_noswz(sf_smem + 512u * (1 + i)));
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // 4 x (K = 32 fp8): 32 bytes per step, like bf16
          const uint64_t ad = smem_desc_sw128(a_addr + k * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_addr + k * 32, 16, 1024);
          tc_mma_mxf8(tmem_d, ad, bd, idesc_mxf8(kTileM, n_mma, k), t_sfa, t_sfb,
                      (ks | k) != 0 ? 1u : 0u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t ad = p.a_mn ? smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(a_addr + k * 32, 16, 1024);
          const uint64_t bd = p.b_mn ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(b_addr + k * 32, 16, 1024);
          tc_mma_bf16(tmem_d, ad, bd, idesc, (ks | k) != 0 ? 1u : 0u);
        }
      }
      tc_commit(&s.empty[stage]);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    tc_commit(&s.tfull[acc]);
  }
  // everything this thread issued must be finished before TMEM is freed
  tc_commit(&s.fin);
  const uint32_t a = smem_u32(&s.fin);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, 0)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      raise_error(p.err, MOE_DEVERR_TIMEOUT);
      break;
    }
  }
}

// ------------------------------------------------------------------ CTA pairs
// A pair of CTAs (a cluster of two) runs one 256 x BN tile with one
// tcgen05.mma.cta_group::2 (M = 256): CTA r holds rows [128 r, 128 r + 128)
// of A and columns [r BN/2, (r + 1) BN/2) of B in its shared memory, and rows
// [128 r, 128 r + 128) of the accumulator in its tensor memory.  The even CTA
// issues the MMAs; the odd CTA's copies complete on the even CTA's `full`
// barriers, the MMA commits arrive on both CTAs' barriers (multicast), and the
// odd CTA's epilogue arrives on the even CTA's `tempty` barrier.

// Tile `t` of the pair schedule, seen from CTA `rank`.  M-grouped: the pair
// covers m-tiles (2j, 2j + 1) of one expert; when the expert has an odd number
// of m-tiles the odd CTA of its last pair reloads the even CTA's rows and
// stores nothing (`valid` false).  K-grouped: m-tiles (2i, 2i + 1), the experts
// taken in the order kgroup_order sets up.
MOE_DEV int total_tiles_pair(const Params& p, const Ctl& s) {
  if (p.mode == MODE_MGROUP) return s.pair_off[p.E] * p.n_tiles;
  return p.E * (p.m_tiles / 2) * p.n_tiles;
}
// Every pair takes one tile of each round of nclusters tiles.  With experts of
// more than twice the mean rows (long tiles), odd rounds run backwards, so the
// pair that got the first (longest) tile of one round gets the last of the next;
// otherwise (pair_off[E] == 0) every round runs forwards.
MOE_DEV int kgroup_snake(const Params& p, const Ctl& s, int t) {
  const int np = (int)gridDim.x / 2;
  const int round = t / np;
  if (!(round & 1)) return t;
  const int n_r = min(np, total_tiles_pair(p, s) - round * np);
  return round * np + (n_r - 1 - (t - round * np));
}

// KG: the kernel runs K-grouped schedules only, else M-grouped ones only (each
// kernel is compiled for one of the two, with no code of the other).
template <bool KG>
MOE_DEV TileInfo decode_pair(const Params& p, const Ctl& s, int t, int rank, bool& valid) {
  TileInfo ti;
  valid = true;
  ti.kb = 0;
  if constexpr (KG) {
    const bool skew = s.pair_off[p.E] > 0;
    if (skew) t = kgroup_snake(p, s, t);
    const int per = (p.m_tiles / 2) * p.n_tiles;
    const int g = t / per;              // the g-th expert of kgroup_order's order
    ti.e = skew ? s.pair_off[g] : g;
    const int r = t - g * per;
    const int pm = r / p.n_tiles;
    ti.n_tile = r - pm * p.n_tiles;
    ti.m_tile = 2 * pm + rank;
    ti.k0row = s.tile_off[ti.e] * kTileM;
    ti.ks = (s.tile_off[ti.e + 1] - s.tile_off[ti.e]) * (kTileM / kBK);
  } else {
    const int pt = t / p.n_tiles;
    ti.n_tile = t - pt * p.n_tiles;
    ti.e = find_group(s.pair_off, p.E, pt);
    const int m = s.tile_off[ti.e] + 2 * (pt - s.pair_off[ti.e]) + rank;
    valid = m < s.tile_off[ti.e + 1];
    ti.m_tile = valid ? m : m - 1;
    ti.k0row = 0;
    ti.ks = p.k_steps;
  }
  return ti;
}

// One stage's copies of this CTA (its A rows and its half of B), counted on
// the even CTA's full barrier (cluster address `fb`).
MOE_DEV void stage_loads_pair(const Params& p, const TileInfo& ti, int ks, int rank, uint8_t* sa,
                              uint32_t fb, const CUtensorMap* tA0, const CUtensorMap* tA1,
                              const CUtensorMap* tB0, const CUtensorMap* tB1) {
  uint8_t* sb = sa + kABytes;
  const int nh = p.BN / 2;                        // this CTA's columns of B
  const int n0 = ti.n_tile * p.BN + rank * nh;
  if (p.mode == MODE_KGROUP) {
    const bool hi = ti.m_tile >= p.m_split;
    const CUtensorMap* ma = hi ? tA1 : tA0;
    const int mcol = (ti.m_tile - (hi ? p.m_split : 0)) * kTileM;
    const int krow = ti.k0row + ks * kBK;
    tma_load_2d_pair(sa, ma, fb, mcol, krow);
    tma_load_2d_pair(sa + kABytes / 2, ma, fb, mcol + 64, krow);
    for (int i = 0; i < nh / 64; ++i) tma_load_2d_pair(sb + i * 8192, tB0, fb, n0 + 64 * i, krow);
    return;
  }
  const bool src1 = ks >= p.k_split;
  const int kk = (src1 ? ks - p.k_split : ks) * kBK;
  const CUtensorMap* mb = src1 ? tB1 : tB0;
  tma_load_2d_pair(sa, src1 ? tA1 : tA0, fb, kk, ti.m_tile * kTileM);
  if (p.b_mn) {
    const int krow = ti.e * p.b_group_rows + kk;
    for (int i = 0; i < nh / 64; ++i) tma_load_2d_pair(sb + i * 8192, mb, fb, n0 + 64 * i, krow);
  } else if (p.b_dual) {   // the even CTA holds the gate rows, the odd CTA the up rows
    tma_load_2d_pair(sb, rank == 0 ? tB0 : tB1, fb, kk, ti.e * p.b_group_rows + ti.n_tile * 128);
  } else {
    tma_load_2d_pair(sb, mb, fb, kk, ti.e * p.b_group_rows + n0);
  }
}

// In-kernel dequantisation: this CTA's copies of one stage.  A goes to the even
// CTA's full barrier as on every pair; the B codes (64 rows x 128 columns) and
// the scale atom that covers them land on this CTA's rawfull barrier.
MOE_DEV void stage_loads_pair_dq(const Params& p, const TileInfo& ti, int ks, int rank,
                                 uint8_t* sa, uint32_t fb, uint64_t* rb, const CUtensorMap* tA0,
                                 const CUtensorMap* tA1, const CUtensorMap* tB0) {
  const bool hi = ti.m_tile >= p.m_split;
  const CUtensorMap* ma = hi ? tA1 : tA0;
  const int mcol = (ti.m_tile - (hi ? p.m_split : 0)) * kTileM;
  const int krow = ti.k0row + ks * kBK;
  tma_load_2d_pair(sa, ma, fb, mcol, krow);
  tma_load_2d_pair(sa + kABytes / 2, ma, fb, mcol + 64, krow);
  const int n0 = ti.n_tile * p.BN + rank * (p.BN / 2);   // a multiple of 128
  mbar_arrive_expect_tx(rb, (uint32_t)(kDqRawBytes + 512));
  tma_load_2d(sa + kABytes, tB0, rb, n0, krow);
  bulk_load(sa + kABytes + kDqRawBytes,
            p.sfq + ((size_t)(krow >> 7) * (size_t)p.sfq_k + (size_t)(n0 >> 7)) * 512u, 512u, rb);
}

// Bounded wait for the last `stages` completions of one barrier array (copies
// still in flight when a CTA gives up).
MOE_DEV void drain_stages(uint64_t* bars, long issued, int stages) {
  for (long i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
    const uint32_t a = smem_u32(&bars[(int)(i % stages)]);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, (uint32_t)((i / stages) & 1))) {
      if (globaltimer() - t0 > kWaitLimitNs) break;
    }
  }
}

template <bool DQB, bool KG>
MOE_DEV void producer_pair(const Params& p, Ctl& s, uint8_t* ring, int rank,
                           const CUtensorMap* tA0, const CUtensorMap* tA1, const CUtensorMap* tB0,
                           const CUtensorMap* tB1) {
  if (p.inject_stall) return;
  const int nt = total_tiles_pair(p, s);
  const int nclusters = (int)gridDim.x / 2;
  const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);   // even CTA's full[0]
  int stage = 0;
  uint32_t phase = 0;
  long issued = 0;
  bool ok = true;
  for (int t = (int)blockIdx.x / 2; ok && t < nt; t += nclusters) {
    bool valid;
    const TileInfo ti = decode_pair<KG>(p, s, t, rank, valid);
    for (int ks = 0; ks < ti.ks; ++ks) {
      if (!mbar_wait(&s.empty[stage], phase ^ 1u, &s.abort, p.err)) { ok = false; break; }
      if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2u * (uint32_t)p.pair_half_bytes);
      ++issued;
      if constexpr (DQB)
        stage_loads_pair_dq(p, ti, ks, rank, ring + stage * p.stage_bytes,
                            full0 + 8u * (uint32_t)stage, &s.rawfull[stage], tA0, tA1, tB0);
      else
        stage_loads_pair(p, ti, ks, rank, ring + stage * p.stage_bytes,
                         full0 + 8u * (uint32_t)stage, tA0, tA1, tB0, tB1);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    // copies in flight land on the even CTA's barriers (and, dequantising, on
    // this CTA's rawfull): the even CTA waits for the stages it armed; both
    // give their copies time to land before leaving
    if (rank == 0) drain_stages(s.full, issued, p.stages);
    if (DQB) drain_stages(s.rawfull, issued, p.stages);
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 100000ull) {}   // 100 us
  }
}

template <bool DQB, bool KG>
MOE_DEV void mma_issuer_pair(const Params& p, Ctl& s, uint8_t* ring, uint32_t tmem_base, int rank) {
  if (rank == 0) {
    uint8_t* slots = ring + p.stages * p.stage_bytes;   // DQB: the converted B tiles
    int slot = 0;
    uint32_t sphase = 0;
    const int nt = total_tiles_pair(p, s);
    const int nclusters = (int)gridDim.x / 2;
    const int n_mma = p.b_dual ? 256 : p.BN;
    const uint32_t idesc = idesc_bf16_f32(2 * kTileM, n_mma, p.a_mn, p.b_mn);
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int t = (int)blockIdx.x / 2; ok && t < nt; t += nclusters, ++it) {
      bool valid;
      const TileInfo ti = decode_pair<KG>(p, s, t, 0, valid);
      const int acc = it % p.num_acc;
      const uint32_t use = (uint32_t)(it / p.num_acc);
      if (!mbar_wait(&s.tempty[acc], (use & 1u) ^ 1u, &s.abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tmem_d = tmem_base + (uint32_t)(acc * p.acc_cols);
      for (int ks = 0; ks < ti.ks; ++ks) {
        if (!mbar_wait(&s.full[stage], phase, &s.abort, p.err)) { ok = false; break; }
        if (DQB && !mbar_wait(&s.bfull[slot], sphase, &s.abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + stage * p.stage_bytes);
        const uint32_t b_addr = DQB ? smem_u32(slots + slot * kDqSlotBytes) : a_addr + kABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          const uint64_t ad = p.a_mn ? smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(a_addr + k * 32, 16, 1024);
          const uint64_t bd = p.b_mn ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(b_addr + k * 32, 16, 1024);
          tc_mma_bf16_pair(tmem_d, ad, bd, idesc, (ks | k) != 0 ? 1u : 0u);
        }
        tc_commit_pair(&s.empty[stage]);
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
        if constexpr (DQB) {
          tc_commit_pair(&s.bempty[slot]);
          if (++slot == kDqSlots) { slot = 0; sphase ^= 1u; }
        }
      }
      if (!ok) break;
      tc_commit_pair(&s.tfull[acc]);
    }
    tc_commit_pair(&s.fin);      // both CTAs learn when the pair's MMAs are done
  }
  const uint32_t a = smem_u32(&s.fin);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, 0)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      raise_error(p.err, MOE_DEVERR_TIMEOUT);
      break;
    }
  }
}

// ------------------------------------------------------------------ epilogues
// Each epilogue thread owns one row of the 128-row tile; `tb` is the TMEM
// address of that row's accumulator (lane field set, column 0).
MOE_DEV void store_bf16x32(__nv_bfloat16* dst, const uint32_t* v) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d4[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                       pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
  }
}

// One MXFP8 block held by one thread: 32 values -> 32 E4M3 codes + 1 scale byte.
// E4M3 codes of one 32-value block: bytes 0-15 in lo, 16-31 in hi; returns
// the block's E8M0 scale byte
MOE_DEV uint32_t mx_quant32_regs(const uint32_t* bits, uint4& lo, uint4& hi) {
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(bits[i]);
    amax = fmaxf(amax, fabsf(v[i]));
  }
  const int sx = mx_scale_exp(amax);
  const float inv = exp2i(-sx);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= inv;
  const uint2 q0 = e4m3x8(v), q1 = e4m3x8(v + 8), q2 = e4m3x8(v + 16), q3 = e4m3x8(v + 24);
  lo = make_uint4(q0.x, q0.y, q1.x, q1.y);
  hi = make_uint4(q2.x, q2.y, q3.x, q3.y);
  return (uint32_t)(sx + 127);
}

// The same, codes stored to `codes` (32 bytes, 16-byte aligned).
MOE_DEV uint32_t mx_quant32(const uint32_t* bits, uint8_t* codes) {
  uint4 lo, hi;
  const uint32_t sb = mx_quant32_regs(bits, lo, hi);
  reinterpret_cast<uint4*>(codes)[0] = lo;
  reinterpret_cast<uint4*>(codes)[1] = hi;
  return sb;
}

MOE_DEV void mx_store32(const uint32_t* bits, uint8_t* codes, uint8_t* sf_byte) {
  *sf_byte = (uint8_t)mx_quant32(bits, codes);
}

// Columns [c0, c1) of the tile, 32 at a time.
MOE_DEV void epilogue_router(const Params& p, const TileInfo& ti, int r, uint32_t tb, int c0,
                             int c1, uint32_t* v) {
  // EPI_ROUTER: fp32 logits (+ bias), rows < T and columns < E only
  // With the K loop split in two, each part adds its sum into the zeroed
  // logits (the first part with the bias): (0 + a) + b == (0 + b) + a, so the
  // result does not depend on which part lands first.  Lane = row: the lanes
  // of a warp touch 32 different rows (cache lines) per access; whole 32-column
  // chunks of rows that start on 16 bytes go out as 4-wide loads, stores and
  // atomics (8 per lane instead of 32).
  const int64_t row = (int64_t)ti.m_tile * kTileM + r;
  float* out = static_cast<float*>(p.out0);
  const bool add_bias = p.bias != nullptr && ti.kb == 0;
  for (int c = c0; c < c1; c += 32) {
    tmem_ld32(tb + c, v);      // warp-collective: executed by every lane
    if (row >= p.m_valid) continue;
    float* o = out + row * p.n_valid + c;
    const float* bz = add_bias ? p.bias + row * p.n_valid + c : nullptr;
    if (p.n_valid % 4 == 0 && c + 32 <= p.n_valid) {
      float4 b4[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        b4[q] = add_bias ? *reinterpret_cast<const float4*>(bz + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 val = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        if (add_bias) {
          val.x += b4[q].x; val.y += b4[q].y; val.z += b4[q].z; val.w += b4[q].w;
        }
        if (p.k_parts > 1)
          atomicAdd(reinterpret_cast<float4*>(o + 4 * q), val);
        else
          *reinterpret_cast<float4*>(o + 4 * q) = val;
      }
    } else {
      for (int i = 0; i < 32 && c + i < p.n_valid; ++i) {
        float val = __uint_as_float(v[i]);
        if (add_bias) val += bz[i];
        if (p.k_parts > 1)
          atomicAdd(o + i, val);
        else
          o[i] = val;
      }
    }
  }
}

// E8M0 scale byte -> 2^(s - 127) as a binary32: the biased exponent field is s
// itself for s >= 1; 2^-127 (s = 0) is the subnormal with only mantissa bit 22.
MOE_DEV float e8m0_value(uint32_t sb) { return __uint_as_float(sb != 0u ? sb << 23 : 0x00400000u); }

// Converter warps (in-kernel dequantisation of B): for every stage in the
// producer's order, wait for this CTA's codes and scales, wait for a free B
// slot, write value = E4M3 code x 2^(scale - 127) rounded to bf16 (the same
// arithmetic as the global dequantisation) into the slot's two 64-column
// halves, 128-byte swizzled, and arrive on the even CTA's bfull barrier.
// Thread i converts 16-byte output chunks i, i + 32 kConvWarps, ... of the 64 x 128
// tile: chunk c is row c / 16, columns 8 (c % 16) .. + 7.
MOE_DEV void converter_pair(const Params& p, Ctl& s, uint8_t* ring, int ctid, int lane) {
  const int nt = total_tiles_pair(p, s);
  const int nclusters = (int)gridDim.x / 2;
  const int rank = (int)cluster_ctarank();
  const uint32_t bfull0 = mapa_shared(smem_u32(&s.bfull[0]), 0);
  uint8_t* slots = ring + p.stages * p.stage_bytes;
  int stage = 0, slot = 0;
  uint32_t phase = 0, sphase = 0;
  for (int t = (int)blockIdx.x / 2; t < nt; t += nclusters) {
    bool valid;
    const TileInfo ti = decode_pair<true>(p, s, t, rank, valid);
    for (int ks = 0; ks < ti.ks; ++ks) {
      bool ok = mbar_wait(&s.rawfull[stage], phase, &s.abort, p.err);
      ok = ok && mbar_wait(&s.bempty[slot], sphase ^ 1u, &s.abort, p.err);
      if (!__all_sync(0xffffffffu, ok)) return;
      const uint8_t* raw = ring + stage * p.stage_bytes + kABytes;
      const uint8_t* sf = raw + kDqRawBytes;
      uint8_t* dst = slots + slot * kDqSlotBytes;
      const int r0 = (ti.k0row + ks * kBK) & 127;   // first row of the stage inside the atom
#pragma unroll 4
      for (int i = 0; i < (kBK * 16) / (32 * kConvWarps); ++i) {
        const int c = ctid + 32 * kConvWarps * i;
        const int r = c >> 4, j = c & 15;
        const uint2 w = *reinterpret_cast<const uint2*>(raw + r * 128 + j * 8);
        const int R = r0 + r;
        const float scale = e8m0_value(sf[(R & 31) * 16 + (R >> 5) * 4 + (j >> 2)]);
        float f[8];
        e4m3x2_to_f32(w.x & 0xFFFFu, f[0], f[1]);
        e4m3x2_to_f32(w.x >> 16, f[2], f[3]);
        e4m3x2_to_f32(w.y & 0xFFFFu, f[4], f[5]);
        e4m3x2_to_f32(w.y >> 16, f[6], f[7]);
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] *= scale;
        *reinterpret_cast<uint4*>(dst + (j >> 3) * 8192 + r * 128 + (((j & 7) ^ (r & 7)) << 4)) =
            pack8(f);
      }
      fence_proxy_async_smem();   // the MMA (async proxy) reads what was just written
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bfull0 + 8u * (uint32_t)slot);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      if (++slot == kDqSlots) { slot = 0; sphase ^= 1u; }
    }
  }
}

// Direct-store epilogues: the router (bf16 kernels) and every MXFP8 epilogue;
// each instantiation compiles only the branches it can reach (register
// pressure at the 168-register cap).
template <bool MX>
MOE_DEV void epilogue_tile(const Params& p, const TileInfo& ti, int r, uint32_t tb, int c0, int c1) {
  uint32_t v[32];
  if (!MX) {
    epilogue_router(p, ti, r, tb, c0, c1, v);
    return;
  }
  if (!MOE_CHECK_OK(ti.m_tile, p.rows_max / kTileM)) return;   // the tile's rows (checks build)
  if (p.epi == EPI_BF16) {
    const int64_t row = (int64_t)ti.m_tile * kTileM + r;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out0) + row * p.ldo + (int64_t)ti.n_tile * p.BN;
    for (int c = c0; c < c1; c += 32) {
      tmem_ld32(tb + c, v);
      store_bf16x32(out + c, v);
    }
  } else if (p.epi == EPI_SWIGLU_FWD_MX) {
    // accumulator columns [0, 64) are H, [64, 128) are U for f columns n_tile*64 + [0, 64)
    const int64_t row = (int64_t)ti.m_tile * kTileM + r;
    const int fc = ti.n_tile * 64;
    const int64_t off = row * p.ldo + fc;
    __nv_bfloat16* H = static_cast<__nv_bfloat16*>(p.out0) + off;
    __nv_bfloat16* U = static_cast<__nv_bfloat16*>(p.out1) + off;
    uint8_t* Aq = static_cast<uint8_t*>(p.out2) + off;
    uint32_t w[32];
    for (int c = c0; c < c1; c += 32) {
      tmem_ld32x2(tb + c, tb + 64 + c, v, w);
      uint32_t a[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        a[i] = __float_as_uint(silu_f(__uint_as_float(v[i])) * __uint_as_float(w[i]));
      store_bf16x32(H + c, v);
      store_bf16x32(U + c, w);
      mx_store32(a, Aq + c, p.osf0 + sf_offset(row, (fc + c) / 32, p.osf_kb));
    }
  } else if (p.epi == EPI_SWIGLU_BWD_MX) {
    const int64_t row = (int64_t)ti.m_tile * kTileM + r;
    const int fc = ti.n_tile * p.BN;
    const int64_t off = row * p.ldo + fc;
    const uint4* H = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.aux0) + off);
    const uint4* U = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.aux1) + off);
    __nv_bfloat16* dH = static_cast<__nv_bfloat16*>(p.out0) + off;
    __nv_bfloat16* dU = static_cast<__nv_bfloat16*>(p.out1) + off;
    uint8_t* dHq = static_cast<uint8_t*>(p.out2) + off;
    uint8_t* dUq = static_cast<uint8_t*>(p.out3) + off;
    for (int c = c0; c < c1; c += 32) {
      uint4 hc[4], uc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        hc[q] = H[c / 8 + q];
        uc[q] = U[c / 8 + q];
      }
      tmem_ld32(tb + c, v);
      uint32_t gh[32], gu[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float h[8], u[8];
        unpack8(hc[q], h);
        unpack8(uc[q], u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float da = __uint_as_float(v[8 * q + i]);
          const float sg = sigmoid_f(h[i]);
          const float si = h[i] * sg;
          const float ds = sg * (1.0f + h[i] * (1.0f - sg));
          gh[8 * q + i] = __float_as_uint(da * u[i] * ds);
          gu[8 * q + i] = __float_as_uint(da * si);
        }
      }
      store_bf16x32(dH + c, gh);
      store_bf16x32(dU + c, gu);
      const size_t so = sf_offset(row, (fc + c) / 32, p.osf_kb);
      mx_store32(gh, dHq + c, p.osf0 + so);
      mx_store32(gu, dUq + c, p.osf1 + so);
    }
  }
}

// ---- epilogue through shared memory: each column half owns a 16 KB buffer of
// 128 rows x 128 bytes in the 128-byte swizzled layout of the output tensor
// maps; thread r fills row r, one elected thread issues the TMA bulk store.
struct OutStager {
  uint8_t* buf;
  int bar_id;
  bool leader;
  int r;
  // the buffer is free once the previous bulk store has read it
  MOE_DEV void begin() const {
    if (leader) bulk_wait_read_all();
    bar_sync(bar_id, kEpiThreads / 2);
  }
  MOE_DEV void put16(int j, const uint4& v) const {   // 128-byte rows, 128-byte swizzle
    *reinterpret_cast<uint4*>(buf + r * 128 + ((j ^ (r & 7)) << 4)) = v;
  }
  // 64-byte rows, 64-byte swizzle; `part` selects one of two 8 KB boxes
  MOE_DEV void put16_r64(int j, const uint4& v, int part) const {
    *reinterpret_cast<uint4*>(buf + part * 8192 + r * 64 + ((j ^ ((r >> 1) & 3)) << 4)) = v;
  }
  // 64 fp32 -> 64 bf16 (128 bytes)
  MOE_DEV void row_bf16(const uint32_t* lo, const uint32_t* hi) const {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      put16(j, make_uint4(pack_bf16x2(__uint_as_float(lo[8 * j]), __uint_as_float(lo[8 * j + 1])),
                          pack_bf16x2(__uint_as_float(lo[8 * j + 2]), __uint_as_float(lo[8 * j + 3])),
                          pack_bf16x2(__uint_as_float(lo[8 * j + 4]), __uint_as_float(lo[8 * j + 5])),
                          pack_bf16x2(__uint_as_float(lo[8 * j + 6]), __uint_as_float(lo[8 * j + 7]))));
#pragma unroll
    for (int j = 0; j < 4; ++j)
      put16(4 + j, make_uint4(pack_bf16x2(__uint_as_float(hi[8 * j]), __uint_as_float(hi[8 * j + 1])),
                              pack_bf16x2(__uint_as_float(hi[8 * j + 2]), __uint_as_float(hi[8 * j + 3])),
                              pack_bf16x2(__uint_as_float(hi[8 * j + 4]), __uint_as_float(hi[8 * j + 5])),
                              pack_bf16x2(__uint_as_float(hi[8 * j + 6]), __uint_as_float(hi[8 * j + 7]))));
  }
  // 32 fp32 (128 bytes)
  MOE_DEV void row_f32(const uint32_t* v) const {
#pragma unroll
    for (int j = 0; j < 8; ++j) put16(j, make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
  }
  MOE_DEV void row_zero() const {
#pragma unroll
    for (int j = 0; j < 8; ++j) put16(j, make_uint4(0, 0, 0, 0));
  }
  MOE_DEV void end(const CUtensorMap* map, int x, int y) const {
    fence_proxy_async_smem();
    bar_sync(bar_id, kEpiThreads / 2);
    if (leader) {
      tma_store_2d(map, buf, x, y);
      bulk_commit();
    }
  }
  // both 8 KB boxes: box 0 to map0, box 1 to map1, at the same coordinates
  MOE_DEV void end2(const CUtensorMap* map0, const CUtensorMap* map1, int x, int y) const {
    fence_proxy_async_smem();
    bar_sync(bar_id, kEpiThreads / 2);
    if (leader) {
      tma_store_2d(map0, buf, x, y);
      tma_store_2d(map1, buf + 8192, x, y);
      bulk_commit();
    }
  }
};

MOE_DEV void silu_mul32(const uint32_t* h, const uint32_t* u, uint32_t* a) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    a[i] = __float_as_uint(silu_f(__uint_as_float(h[i])) * __uint_as_float(u[i]));
}

// 8 columns of dH = dA * U * silu'(H) and dU = dA * silu(H), packed to bf16
MOE_DEV void swiglu_bwd8(const uint32_t* da, const uint4& hq, const uint4& uq, uint4& dh,
                         uint4& du) {
  float h[8], u[8], gh[8], gu[8];
  unpack8(hq, h);
  unpack8(uq, u);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = __uint_as_float(da[i]);
    const float sg = sigmoid_f(h[i]);
    gh[i] = a * u[i] * (sg * (1.0f + h[i] * (1.0f - sg)));
    gu[i] = a * (h[i] * sg);
  }
  dh = pack8(gh);
  du = pack8(gu);
}

// Columns [c0, c1) of the tile through the stager (bf16 outputs 64 columns per
// store, fp32 outputs 32 columns per store).
// F32_ONLY: the instantiation serves weight gradients alone (EPI_F32).
template <bool F32_ONLY>
MOE_DEV void epilogue_tile_tma(const Params& p, const TileInfo& ti, uint32_t tb, int c0, int c1,
                               const OutStager& st, const CUtensorMap* tO0,
                               const CUtensorMap* tO1, const CUtensorMap* tO2) {
  uint32_t v0[32], v1[32];
  const int y = ti.m_tile * kTileM;
  if (!F32_ONLY && p.epi == EPI_BF16) {
    const int xb = ti.n_tile * p.BN;
    for (int c = c0; c < c1; c += 64) {
      tmem_ld32x2(tb + c, tb + c + 32, v0, v1);
      st.begin();
      st.row_bf16(v0, v1);
      st.end(tO0, xb + c, y);
    }
  } else if (!F32_ONLY && p.epi == EPI_SWIGLU_FWD) {
    // accumulator columns [0, 128) are H, [128, 256) are U
    const int xb = ti.n_tile * 128;
    for (int c = c0; c < c1; c += 64) {
      tmem_ld32x2(tb + c, tb + c + 32, v0, v1);              // H
      st.begin();
      st.row_bf16(v0, v1);
      st.end(tO0, xb + c, y);
      tmem_ld32x2(tb + 128 + c, tb + 128 + c + 32, v0, v1);  // U
      st.begin();
      st.row_bf16(v0, v1);
      st.end(tO1, xb + c, y);
      // A = silu(H) * U, H re-read from tensor memory 32 columns at a time
      uint32_t h[32];
      st.begin();
      tmem_ld32(tb + c, h);
      silu_mul32(h, v0, h);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st.put16(j, make_uint4(pack_bf16x2(__uint_as_float(h[8 * j]), __uint_as_float(h[8 * j + 1])),
                               pack_bf16x2(__uint_as_float(h[8 * j + 2]), __uint_as_float(h[8 * j + 3])),
                               pack_bf16x2(__uint_as_float(h[8 * j + 4]), __uint_as_float(h[8 * j + 5])),
                               pack_bf16x2(__uint_as_float(h[8 * j + 6]), __uint_as_float(h[8 * j + 7]))));
      tmem_ld32(tb + c + 32, h);
      silu_mul32(h, v1, h);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st.put16(4 + j, make_uint4(pack_bf16x2(__uint_as_float(h[8 * j]), __uint_as_float(h[8 * j + 1])),
                                   pack_bf16x2(__uint_as_float(h[8 * j + 2]), __uint_as_float(h[8 * j + 3])),
                                   pack_bf16x2(__uint_as_float(h[8 * j + 4]), __uint_as_float(h[8 * j + 5])),
                                   pack_bf16x2(__uint_as_float(h[8 * j + 6]), __uint_as_float(h[8 * j + 7]))));
      st.end(tO2, xb + c, y);
    }
  } else if (!F32_ONLY && p.epi == EPI_SWIGLU_BWD) {
    const int xb = ti.n_tile * p.BN;
    const int64_t off = (int64_t)(y + st.r) * p.ldo + xb;
    const uint4* H = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.aux0) + off);
    const uint4* U = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.aux1) + off);
    // 32 columns per round; the output maps have 64-byte boxes (64-byte swizzle)
    uint4 hq[4], uq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hq[q] = H[c0 / 8 + q];
      uq[q] = U[c0 / 8 + q];
    }
    // one round per 32 columns: dH into box 0, dU into box 1 of the half's buffer
    for (int c = c0; c < c1; c += 32) {
      tmem_ld32(tb + c, v0);   // dA
      st.begin();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 gh, gu;
        swiglu_bwd8(v0 + 8 * q, hq[q], uq[q], gh, gu);
        st.put16_r64(q, gh, 0);
        st.put16_r64(q, gu, 1);
      }
      if (c + 32 < c1) {        // next columns' H and U, loaded while the stores drain
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hq[q] = H[(c + 32) / 8 + q];
          uq[q] = U[(c + 32) / 8 + q];
        }
      }
      st.end2(tO0, tO1, xb + c, y);
    }
  } else {  // EPI_F32: weight gradients, fp32 [E * M, N]
    const bool hi = ti.m_tile >= p.m_split;
    const int yy = (int)(ti.e * p.out_rows_per_group) + (ti.m_tile - (hi ? p.m_split : 0)) * kTileM;
    const CUtensorMap* map = hi ? tO1 : tO0;
    const int xb = ti.n_tile * p.BN;
    for (int c = c0; c < c1; c += 32) {
      if (ti.ks != 0) tmem_ld32(tb + c, v0);
      st.begin();
      if (ti.ks != 0) st.row_f32(v0); else st.row_zero();
      st.end(map, xb + c, yy);
    }
  }
}

template <bool MX, bool PAIR, bool DQB, bool KG>
MOE_DEV void epilogue(const Params& p, Ctl& s, uint32_t tmem_base, int warp, int lane,
                      uint8_t* stage_out, const CUtensorMap* tO0, const CUtensorMap* tO1,
                      const CUtensorMap* tO2, int rank) {
  const int nt = PAIR ? total_tiles_pair(p, s) : total_tiles(p, s.tile_off);
  const int t_first = PAIR ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int t_step = PAIR ? (int)gridDim.x / 2 : (int)gridDim.x;
  // the pair's accumulator-empty barriers live in the even CTA
  const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(&s.tempty[0]), 0) : 0u;
  const int quarter = warp & 3;            // TMEM lanes this warp may access
  const int half = (warp - 2) >> 2;        // which half of the tile's columns
  const int r = quarter * 32 + lane;
  // column range of this warp: half of the tile (of the H half for SwiGLU)
  const int width = (p.epi == EPI_SWIGLU_FWD) ? 128 : (p.epi == EPI_SWIGLU_FWD_MX ? 64 : p.BN);
  int c0, c1;
  if (width >= 64) {
    c0 = half * (width / 2);
    c1 = c0 + width / 2;
  } else {                                 // narrow router tile: first half only
    c0 = 0;
    c1 = (half == 0) ? width : 0;
  }
  OutStager st;
  st.buf = stage_out + half * kStageOutBytes;
  st.bar_id = 1 + half;
  st.leader = (quarter == 2) && (lane == 0);   // first warp of the half (warp 2 or 6)
  st.r = r;
  int it = 0;
  for (int t = t_first; t < nt; t += t_step, ++it) {
    bool valid = true;
    const TileInfo ti = PAIR ? decode_pair<KG>(p, s, t, rank, valid) : decode_tile(p, s.tile_off, t);
    const int acc = it % p.num_acc;
    const uint32_t use = (uint32_t)(it / p.num_acc);
    bool ok = mbar_wait(&s.tfull[acc], use & 1u, &s.abort, p.err);
    // the half's named barriers below need all four of its warps: leave together
    if (p.tma_store) ok = bar_and(st.bar_id, kEpiThreads / 2, ok);
    if (!ok) break;
    tc_fence_after();
    const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * p.acc_cols);
    // a column half past N (the last tile when N = 128 mod 256) is neither
    // read nor written: its operands were zero-filled, its output is clipped
    if (valid && (p.n_cols == 0 || ti.n_tile * p.BN + c0 < p.n_cols)) {
      if (DQB || (!MX && p.tma_store))
        epilogue_tile_tma<DQB>(p, ti, tb, c0, c1, st, tO0, tO1, tO2);
      else
        epilogue_tile<MX>(p, ti, r, tb, c0, c1);
    }
    tc_fence_before();
    if (PAIR)
      mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
    else
      mbar_arrive(&s.tempty[acc]);
  }
  if (st.leader) bulk_wait_all();   // stores complete before the CTA exits
}

// K-grouped pair tiles: the number of long experts (pair_off[E]) and, if there
// are any, the expert order of the schedule (pair_off[0..E-1]; else id order);
// every thread of the CTA calls it
__device__ __noinline__ void kgroup_order(const Params& p, Ctl& s) {
  // weight gradients: a tile's main loop runs over its expert's rows.  The
  // experts with more than twice the mean rows go first, most rows first (the
  // lower id on ties), so that no long tile starts last; the others keep their
  // id order, which mixes short store-bound tiles with longer ones.
  // pair_off[E] keeps the number of such experts.
  const int total = s.tile_off[p.E] - s.tile_off[0];
  int mine = 0;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x)
    mine += ((s.tile_off[e + 1] - s.tile_off[e]) * p.E > 2 * total) ? 1 : 0;
  static_assert(kMaxE <= kThreads, "one expert per thread at most");
  const int nh = __syncthreads_count(mine);
  for (int e = threadIdx.x; e < p.E && nh > 0; e += blockDim.x) {
    const int ke = s.tile_off[e + 1] - s.tile_off[e];
    const bool heavy_e = ke * p.E > 2 * total;
    int g = 0;
    for (int o = 0; o < p.E; ++o) {
      const int ko = s.tile_off[o + 1] - s.tile_off[o];
      const bool heavy_o = ko * p.E > 2 * total;
      if (heavy_e)
        g += (heavy_o && (ko > ke || (ko == ke && o < e))) ? 1 : 0;
      else
        g += (!heavy_o && o < e) ? 1 : 0;
    }
    s.pair_off[heavy_e ? g : nh + g] = e;
  }
  if (threadIdx.x == 0) s.pair_off[p.E] = nh;
}

// KG (CTA pairs): compiled for K-grouped schedules (weight gradients) only, else
// for M-grouped ones only; the dequantising kernel (DQB) is K-grouped.
template <bool MX, bool PAIR, bool DQB = false, bool KG = DQB>
__global__ void __launch_bounds__(DQB ? kThreadsDq : kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tA0,
                        const __grid_constant__ CUtensorMap tA1,
                        const __grid_constant__ CUtensorMap tB0,
                        const __grid_constant__ CUtensorMap tB1,
                        const __grid_constant__ CUtensorMap tO0,
                        const __grid_constant__ CUtensorMap tO1,
                        const __grid_constant__ CUtensorMap tO2, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {   // uniform over the grid: report and leave
    pdl_wait();
    if (threadIdx.x == 0) raise_error(p.err, MOE_DEVERR_BOUNDS);
    return;
  }
  uint8_t* ring = smem_raw;
  uint8_t* stage_out = ring + kRingBytes;
  Ctl& s = *reinterpret_cast<Ctl*>(stage_out + 2 * kStageOutBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);
      mbar_init(&s.tempty[i], PAIR ? 2 * kEpiThreads : kEpiThreads);
    }
    if (DQB) {
      for (int i = 0; i < p.stages; ++i) mbar_init(&s.rawfull[i], 1);
      for (int i = 0; i < kDqSlots; ++i) {
        mbar_init(&s.bfull[i], 2 * kConvWarps);   // one arrival per converter warp of the pair
        mbar_init(&s.bempty[i], 1);
      }
    }
    mbar_init(&s.fin, 1);
    s.abort = 0;
    fence_barrier_init();
  }
  pdl_wait();   // the previous kernel's outputs (operands, tile_offsets) are visible from here
  if (p.mode != MODE_DENSE) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s.tile_off[i] = p.tile_offsets[i];
  }
  if (PAIR) {
    __syncthreads();
    if constexpr (KG) {
      kgroup_order(p, s);
    } else if (threadIdx.x == 0) {
      int run = 0;
      for (int e = 0; e < p.E; ++e) {
        s.pair_off[e] = run;
        run += (s.tile_off[e + 1] - s.tile_off[e] + 1) / 2;
      }
      s.pair_off[p.E] = run;
    }
    cluster_sync();   // both CTAs' barriers are initialised before any remote arrive
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tA0);
    prefetch_tensormap(&tA1);
    prefetch_tensormap(&tB0);
    prefetch_tensormap(&tB1);
    if (p.tma_store) {
      prefetch_tensormap(&tO0);
      prefetch_tensormap(&tO1);
      prefetch_tensormap(&tO2);
    }
  }
  if (warp == 1) {
    if (PAIR)
      tmem_alloc_pair(&s.tmem_base, (uint32_t)p.tmem_cols);
    else
      tmem_alloc(&s.tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      if (PAIR)
        producer_pair<DQB, KG>(p, s, ring, rank, &tA0, &tA1, &tB0, &tB1);
      else
        producer<MX>(p, s, ring, &tA0, &tA1, &tB0, &tB1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (PAIR)
        mma_issuer_pair<DQB, KG>(p, s, ring, tmem_base, rank);
      else
        mma_issuer<MX>(p, s, ring, tmem_base);
    }
  } else if (warp < kThreads / 32) {
    epilogue<MX, PAIR, DQB, KG>(p, s, tmem_base, warp, lane, stage_out, &tO0, &tO1, &tO2, rank);
  } else if (DQB && PAIR) {
    converter_pair(p, s, ring, (int)threadIdx.x - kThreads, lane);
  }

  tc_fence_before();
  if (PAIR)
    cluster_sync();   // the partner no longer reads this CTA's memory
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ MXFP8 on CTA pairs
// One 256 x 256 tile per pair with tcgen05.mma.cta_group::2.kind::mxf8f6f4
// (M = 256, N = 256, K = 32 per instruction, 4 per 128-byte stage).  Each CTA
// stages, per K step of 128 codes: its 128 A rows, its 128 of the tile's 256 B
// rows, the 512-byte scale atom of its A rows and both scale atoms of the B
// rows (every CTA needs the B scales of all N columns); all of it lands on the
// even CTA's `full` barrier (.cta_group::2 TMA, the scales through a 2-D byte
// view of the atom array).  The even CTA copies the stage's scale atoms to
// tensor memory (tcgen05.cp.cta_group::2: each CTA's atoms to its own tensor
// memory) and issues the MMAs.  Tensor memory: one 256-column accumulator,
// then a ring of scale columns (16 per stage: A at +0, B at +4 and +8).  The
// accumulator is single: the epilogue reads its 128 columns into registers,
// releases the accumulator and only then computes and stores, so the next
// tile's main loop overlaps all but the tensor-memory reads.
// 384 threads in three warpgroups: warpgroup 0 (warp 0 producer, warp 1 MMA
// issuer, warps 2-3 idle) gives registers back with setmaxnreg.dec, the two
// epilogue warpgroups (warps 4-11, warp w on tensor-memory lane quarter w % 4,
// column half (w - 4) / 4) take them with setmaxnreg.inc: 128 fp32 accumulator
// values per thread stay in registers without spilling.
// Register budget: launched at 168 per thread (384 x 168 = 64512 per CTA),
// 128 x 80 + 256 x 208 = 63488 after the split; per SM sub-partition
// (three warps) 32 x (80 + 2 x 208) = 15872 <= 16384.
constexpr int kMxPairThreads = 384;
constexpr int kMxPairLaunchRegs = 168;
constexpr int kMxPairRoleRegs = 80;
constexpr int kMxPairEpiRegs = 208;
static_assert(128 * kMxPairRoleRegs + 256 * kMxPairEpiRegs <= kMxPairThreads * kMxPairLaunchRegs,
              "setmaxnreg split exceeds the launch allocation");
static_assert(32 * (kMxPairRoleRegs + 2 * kMxPairEpiRegs) <= 16384, "sub-partition registers");
constexpr int kMxPairBN = 256;
constexpr int kMxCodeBytes = kTileM * 128;                   // 128 rows x 128 E4M3 codes
constexpr int kMxPairSfOff = 2 * kMxCodeBytes;               // scale atoms after A and B
constexpr int kMxPairTx = 2 * kMxCodeBytes + 3 * 512;        // one CTA's bytes per stage
constexpr int kMxPairStageBytes = (kMxPairTx + 1023) & ~1023;
// the TMA-store staging buffers are not used by these epilogues: the ring takes them
constexpr int kMxPairStages = (kRingBytes + 2 * kStageOutBytes) / kMxPairStageBytes;
constexpr uint32_t kMxSfCol0 = 256;
constexpr uint32_t kMxSfColsPerStage = 16;
// bf16 outputs leave through shared memory and TMA bulk stores, 32 columns at a
// time: one 8 KB buffer (128 rows x 64 bytes, 64-byte swizzle) per column half,
// after the ring
constexpr int kMxStageHalfBytes = kTileM * 64;
static_assert(kMxPairStages * kMxPairStageBytes + 2 * kMxStageHalfBytes <=
                  kRingBytes + 2 * kStageOutBytes, "MXFP8 pair shared memory");
// The SwiGLU backward also reads H and U: each half has one set of (H, U)
// 32-column chunks (8 KB each, the output layout), TMA-loaded as soon as the
// previous chunk has left; dH and dU overwrite them in place and leave by TMA
// store.  A 5-stage ring makes room (measured on 8 experts x 4096 rows,
// d = 4096, f = 2048: 4 stages with two sets per half 0.278 ms, 5 stages with
// one set 0.255 ms: the main loop waited for operands 30 % of its time).
constexpr int kMxBwdStages = 5;
constexpr int kMxHuSetBytes = 2 * kTileM * 64;
constexpr int kMxHuHalfBytes = kMxHuSetBytes;
// Their E4M3 codes leave the same way: per half one buffer of dH codes and one
// of dU codes, 128 rows x 32 bytes each (32-byte swizzle), after the H/U sets.
constexpr int kMxCodeHalfBytes = 2 * kTileM * 32;
static_assert(kMxBwdStages * kMxPairStageBytes + 2 * kMxHuHalfBytes + 2 * kMxCodeHalfBytes <=
                  kRingBytes + 2 * kStageOutBytes, "MXFP8 pair backward shared memory");
static_assert(kMxPairStages >= 4 && kMxPairStages <= kMaxStages, "MXFP8 pair ring depth");
static_assert(kMxSfCol0 + kMxSfColsPerStage * kMxPairStages <= kTmemCols, "MXFP8 pair TMEM");

struct MxMaps {           // A, B and their scale-atom views, sources 0 and 1
  const CUtensorMap* a[2];
  const CUtensorMap* b[2];
  const CUtensorMap* sa[2];
  const CUtensorMap* sb[2];
};

// One stage's copies of this CTA, counted on the even CTA's full barrier.
MOE_DEV void stage_loads_mx_pair(const Params& p, const TileInfo& ti, int ks, int rank, uint8_t* sa,
                                 uint32_t fb, const MxMaps& mp) {
  const int src = ks >= p.k_split ? 1 : 0;
  const int kk = (src ? ks - p.k_split : ks) * 128;
  const int brow = ti.e * p.b_group_rows + ti.n_tile * kMxPairBN;   // first B row of the tile
  tma_load_2d_pair(sa, mp.a[src], fb, kk, ti.m_tile * kTileM);
  tma_load_2d_pair(sa + kMxCodeBytes, mp.b[src], fb, kk, brow + rank * kTileM);
  uint8_t* sf = sa + kMxPairSfOff;
  // atom views: two 256-byte rows per 512-byte atom
  tma_load_2d_pair(sf, mp.sa[src], fb, 0, 2 * (ti.m_tile * p.sf_ka + kk / 128));
  tma_load_2d_pair(sf + 512, mp.sb[src], fb, 0, 2 * ((brow >> 7) * p.sf_kb + kk / 128));
  tma_load_2d_pair(sf + 1024, mp.sb[src], fb, 0, 2 * (((brow >> 7) + 1) * p.sf_kb + kk / 128));
}

MOE_DEV void producer_mx_pair(const Params& p, Ctl& s, uint8_t* ring, int rank, const MxMaps& mp) {
  if (p.inject_stall) return;
  const int nt = total_tiles_pair(p, s);
  const int nclusters = (int)gridDim.x / 2;
  const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);   // even CTA's full[0]
  int stage = 0;
  uint32_t phase = 0;
  long issued = 0;
  bool ok = true;
  for (int t = (int)blockIdx.x / 2; ok && t < nt; t += nclusters) {
    bool valid;
    const TileInfo ti = decode_pair<false>(p, s, t, rank, valid);
    for (int ks = 0; ks < ti.ks; ++ks) {
      if (!mbar_wait(&s.empty[stage], phase ^ 1u, &s.abort, p.err)) { ok = false; break; }
      if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2u * (uint32_t)kMxPairTx);
      ++issued;
      stage_loads_mx_pair(p, ti, ks, rank, ring + stage * p.stage_bytes,
                          full0 + 8u * (uint32_t)stage, mp);
      if (++stage == p.stages) { stage = 0; phase ^= 1u; }
    }
  }
  if (!ok) {
    if (rank == 0) drain_stages(s.full, issued, p.stages);
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 100000ull) {}   // 100 us for the odd CTA's copies to land
  }
}

MOE_DEV void mma_issuer_mx_pair(const Params& p, Ctl& s, uint8_t* ring, uint32_t tmem_base,
                                int rank) {
  if (rank == 0) {
    const int nt = total_tiles_pair(p, s);
    const int nclusters = (int)gridDim.x / 2;
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int t = (int)blockIdx.x / 2; ok && t < nt; t += nclusters, ++it) {
      bool valid;
      const TileInfo ti = decode_pair<false>(p, s, t, 0, valid);
      if (!mbar_wait(&s.tempty[0], ((uint32_t)it & 1u) ^ 1u, &s.abort, p.err)) { ok = false; break; }
      tc_fence_after();
      for (int ks = 0; ks < ti.ks; ++ks) {
        if (!mbar_wait(&s.full[stage], phase, &s.abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(ring + stage * p.stage_bytes);
        const uint32_t b_addr = a_addr + kMxCodeBytes;
        const uint32_t sf = a_addr + kMxPairSfOff;
        const uint32_t t_sfa = tmem_base + kMxSfCol0 + (uint32_t)stage * kMxSfColsPerStage;
        const uint32_t t_sfb = t_sfa + 4u;
        tc_cp_32x128b_x4_pair(t_sfa, smem_desc_noswz(sf));
        tc_cp_32x128b_x4_pair(t_sfb, smem_desc_noswz(sf + 512u));
        tc_cp_32x128b_x4_pair(t_sfb + 4u, smem_desc_noswz(sf + 1024u));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = smem_desc_sw128(a_addr + k * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_addr + k * 32, 16, 1024);
          tc_mma_mxf8_pair(tmem_base, ad, bd, idesc_mxf8(2 * kTileM, kMxPairBN, k), t_sfa, t_sfb,
                           (ks | k) != 0 ? 1u : 0u);
        }
        tc_commit_pair(&s.empty[stage]);
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit_pair(&s.tfull[0]);
    }
    tc_commit_pair(&s.fin);
  }
  const uint32_t a = smem_u32(&s.fin);
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(a, 0)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      raise_error(p.err, MOE_DEVERR_TIMEOUT);
      break;
    }
  }
}

// Output staging of one column half (four warps, 128 rows): 64-byte rows,
// 64-byte swizzle, stored by one elected thread with a TMA bulk store.
struct MxStager {
  uint8_t* buf;
  int bar_id;
  bool leader;
  int r;
  MOE_DEV void begin() const {   // the previous bulk store has read the buffer
    if (leader) bulk_wait_read_all();
    bar_sync(bar_id, kEpiThreads / 2);
  }
  MOE_DEV void put16(int j, uint4 v) const {   // 16 raw bytes: granule j of row r
    *reinterpret_cast<uint4*>(buf + r * 64 + ((j ^ ((r >> 1) & 3)) << 4)) = v;
  }
  MOE_DEV void put32(const uint32_t* v) const {   // 32 fp32 -> 32 bf16 of row r
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(buf + r * 64 + ((j ^ ((r >> 1) & 3)) << 4)) =
          make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                     pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                     pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                     pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
  }
  MOE_DEV void end(const CUtensorMap* map, int x, int y) const {
    fence_proxy_async_smem();
    bar_sync(bar_id, kEpiThreads / 2);
    if (leader) {
      tma_store_2d(map, buf, x, y);
      bulk_commit();
    }
  }
  MOE_DEV void store32(const uint32_t* v, const CUtensorMap* map, int x, int y) const {
    begin();
    put32(v);
    end(map, x, y);
  }
};

// Thread (lane quarter q, column half h) owns accumulator row 32q + lane,
// columns [128h, 128h + 128).  bf16 outputs and E4M3 codes leave through
// shared memory and TMA stores (maps tO0, tO1: bf16 outputs; SwiGLU forward:
// tQ1 = A's codes, tQ0 = A dequantised), E8M0 scales by direct stores.
MOE_DEV void epilogue_mx_pair(const Params& p, Ctl& s, uint32_t tmem_base, int warp, int lane,
                              int rank, uint8_t* stage_base, const CUtensorMap* tO0,
                              const CUtensorMap* tO1, const CUtensorMap* tQ0,
                              const CUtensorMap* tQ1) {
  const int nt = total_tiles_pair(p, s);
  const uint32_t tempty0 = mapa_shared(smem_u32(&s.tempty[0]), 0);
  const int quarter = warp & 3;
  const int half = (warp - 4) >> 2;
  const int r = quarter * 32 + lane;
  const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(128 * half);
  const bool bwd = p.epi == EPI_SWIGLU_BWD_MX;
  MxStager st;
  st.buf = stage_base + half * (bwd ? kMxHuHalfBytes : kMxStageHalfBytes);
  st.bar_id = 1 + half;
  st.leader = (warp == 4 + 4 * half) && (lane == 0);
  st.r = r;
  uint64_t* hu_full = &s.hufull[half];
  uint64_t* hu_written = &s.huwritten[half];
  uint32_t vt = 0;   // valid tiles done (SwiGLU backward: the sets' use count)
  int it = 0;
  for (int t = (int)blockIdx.x / 2; t < nt; t += (int)gridDim.x / 2, ++it) {
    bool valid;
    const TileInfo ti = decode_pair<false>(p, s, t, rank, valid);
    valid = valid && MOE_CHECK_OK(ti.m_tile, p.rows_max / kTileM);   // the tile's rows (checks build)
    bool ok = mbar_wait(&s.tfull[0], (uint32_t)it & 1u, &s.abort, p.err);
    // the half's named barriers below need all four of its warps: leave together
    if (!bar_and(st.bar_id, kEpiThreads / 2, ok)) break;
    tc_fence_after();
    uint32_t v[128];
    tmem_ld32x2(tb, tb + 32, v, v + 32);
    tmem_ld32x2(tb + 64, tb + 96, v + 64, v + 96);
    tc_fence_before();
    mbar_arrive_cluster(tempty0);   // the next tile's MMAs may overwrite the accumulator
    if (!valid) continue;
    const int y = ti.m_tile * kTileM;
    const int64_t row = (int64_t)y + r;
    if (p.epi == EPI_BF16) {
      const int x0 = ti.n_tile * kMxPairBN + 128 * half;
#pragma unroll
      for (int c = 0; c < 4; ++c) st.store32(v + 32 * c, tO0, x0 + 32 * c, y);
    } else if (p.epi == EPI_SWIGLU_FWD_MX) {
      // columns [0, 64) of the half are W_gate rows, [64, 128) the matching W_up rows:
      // f columns n_tile * 128 + 64 * half + [0, 64)
      const int fc = ti.n_tile * 128 + 64 * half;
      st.store32(v, tO0, fc, y);
      st.store32(v + 32, tO0, fc + 32, y);
      st.store32(v + 64, tO1, fc, y);
      st.store32(v + 96, tO1, fc + 32, y);
#pragma unroll
      for (int i = 0; i < 64; ++i)
        v[i] = __float_as_uint(silu_f(__uint_as_float(v[i])) * __uint_as_float(v[64 + i]));
      // A's blocks fc/32 and fc/32 + 1 (fc/32 even): adjacent scale bytes, one
      // store; the row's 64 code bytes through the stager
      uint4 q[4];
      const uint32_t s0 = mx_quant32_regs(v, q[0], q[1]), s1 = mx_quant32_regs(v + 32, q[2], q[3]);
      *reinterpret_cast<uint16_t*>(p.osf0 + sf_offset(row, fc / 32, p.osf_kb)) =
          (uint16_t)(s0 | (s1 << 8));
      st.begin();
#pragma unroll
      for (int j = 0; j < 4; ++j) st.put16(j, q[j]);
      st.end(tQ1, fc, y);
      if (p.out3 != nullptr) {
        // A dequantised for the weight gradient: code value x 2^(scale - 127),
        // rounded to bf16, as the dequantiser computes it
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float sc = exp2i((int)(b ? s1 : s0) - 127);
          const uint32_t w[8] = {q[2 * b].x, q[2 * b].y, q[2 * b].z, q[2 * b].w,
                                 q[2 * b + 1].x, q[2 * b + 1].y, q[2 * b + 1].z, q[2 * b + 1].w};
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float lo0, hi0, lo1, hi1;
            e4m3x2_to_f32(w[u] & 0xFFFFu, lo0, hi0);
            e4m3x2_to_f32(w[u] >> 16, lo1, hi1);
            v[64 + 4 * u + 0] = __float_as_uint(lo0 * sc);
            v[64 + 4 * u + 1] = __float_as_uint(hi0 * sc);
            v[64 + 4 * u + 2] = __float_as_uint(lo1 * sc);
            v[64 + 4 * u + 3] = __float_as_uint(hi1 * sc);
          }
          st.store32(v + 64, tQ0, fc + 32 * b, y);
        }
      }
    } else {   // EPI_SWIGLU_BWD_MX: dA for f columns n_tile * 256 + 128 * half + [0, 128)
      const int fc = ti.n_tile * kMxPairBN + 128 * half;
      uint8_t* cbuf = stage_base + 2 * kMxHuHalfBytes + half * kMxCodeHalfBytes;
      uint32_t sh = 0, su = 0;   // the four blocks' scale bytes (fc/32 is a multiple of 4)
      bool fine = true;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint8_t* hb = st.buf;
        uint8_t* ub = hb + kMxHuSetBytes / 2;
        // chunk c is use 4 vt + c of the half's set
        const uint32_t u = 4u * vt + (uint32_t)c;
        fine = fine && mbar_wait(hu_full, u & 1u, &s.abort, p.err);
        uint32_t gu[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int so16 = r * 64 + ((q ^ ((r >> 1) & 3)) << 4);
          float h[8], u[8], gh[8], g2[8];
          unpack8(*reinterpret_cast<const uint4*>(hb + so16), h);
          unpack8(*reinterpret_cast<const uint4*>(ub + so16), u);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float da = __uint_as_float(v[32 * c + 8 * q + i]);
            const float sg = sigmoid_f(h[i]);
            gh[i] = da * u[i] * (sg * (1.0f + h[i] * (1.0f - sg)));
            g2[i] = da * (h[i] * sg);
            v[32 * c + 8 * q + i] = __float_as_uint(gh[i]);
            gu[8 * q + i] = __float_as_uint(g2[i]);
          }
          *reinterpret_cast<uint4*>(hb + so16) = pack8(gh);   // dH, dU over H, U
          *reinterpret_cast<uint4*>(ub + so16) = pack8(g2);
        }
        // this row's E4M3 codes of dH and dU (32 bytes each) into the half's code
        // buffer, once the stores of the previous chunk have read it
        uint4 hl, hh, ul, uh;
        sh |= mx_quant32_regs(v + 32 * c, hl, hh) << (8 * c);
        su |= mx_quant32_regs(gu, ul, uh) << (8 * c);
        const uint32_t g = 4u * vt + (uint32_t)c;
        if (g > 0) fine = fine && mbar_wait(&s.codefree[half], (g - 1u) & 1u, &s.abort, p.err);
        const int sw = (r >> 2) & 1;   // 32-byte swizzle: granule ^= row bit 2
        *reinterpret_cast<uint4*>(cbuf + r * 32 + 16 * sw) = hl;
        *reinterpret_cast<uint4*>(cbuf + r * 32 + 16 * (1 ^ sw)) = hh;
        *reinterpret_cast<uint4*>(cbuf + kTileM * 32 + r * 32 + 16 * sw) = ul;
        *reinterpret_cast<uint4*>(cbuf + kTileM * 32 + r * 32 + 16 * (1 ^ sw)) = uh;
        fence_proxy_async_smem();
        mbar_arrive(hu_written);   // the half's mover stores dH, dU, the codes and refills the set
      }
      const size_t so = sf_offset(row, fc / 32, p.osf_kb);
      *reinterpret_cast<uint32_t*>(p.osf0 + so) = sh;
      *reinterpret_cast<uint32_t*>(p.osf1 + so) = su;
      (void)fine;   // a wait that ran out has set the error word and the abort flag
      ++vt;
    }
  }
  if (st.leader) bulk_wait_all();   // stores complete before the CTA exits
}

// MXFP8 SwiGLU backward: one thread per column half (lane 0 of warp 2 + half)
// moves H and U chunks (32 columns x 128 rows each) into the half's set and
// dH, dU and their E4M3 codes out of the set and the half's code buffer, so
// that the epilogue warps never wait for a bulk copy to read shared memory.
// The set holds chunks 0-3 of each of the CTA's valid tiles in turn; its g-th
// use completes phase g of hufull (H, U landed) and then of huwritten (the
// half's 128 epilogue threads wrote dH, dU over them and the chunk's codes into
// the code buffer); phase g of codefree completes when the g-th chunk's stores
// have read the set and the code buffer.  One copy is in flight at most.
MOE_DEV void hu_mover_mx_pair(const Params& p, Ctl& s, int rank, int half, uint8_t* stage_base,
                              const CUtensorMap* tO0, const CUtensorMap* tO1,
                              const CUtensorMap* tH, const CUtensorMap* tU,
                              const CUtensorMap* tQ0, const CUtensorMap* tQ1) {
  const int nt = total_tiles_pair(p, s);
  const int step = (int)gridDim.x / 2;
  uint8_t* set = stage_base + half * kMxHuHalfBytes;
  uint8_t* cbuf = stage_base + 2 * kMxHuHalfBytes + half * kMxCodeHalfBytes;
  uint64_t* full = &s.hufull[half];
  uint64_t* written = &s.huwritten[half];
  // the next valid tile at or after t, with its first column and row
  auto next_valid = [&](int t, int& fc, int& y) -> int {
    for (; t < nt; t += step) {
      bool valid;
      const TileInfo ti = decode_pair<false>(p, s, t, rank, valid);
      if (valid && MOE_CHECK_OK(ti.m_tile, p.rows_max / kTileM)) {
        fc = ti.n_tile * kMxPairBN + 128 * half;
        y = ti.m_tile * kTileM;
        return t;
      }
    }
    return nt;
  };
  uint32_t loads = 0;
  auto load = [&](int x, int y) {
    mbar_arrive_expect_tx(full, (uint32_t)kMxHuSetBytes);
    tma_load_2d(set, tH, full, x, y);
    tma_load_2d(set + kMxHuSetBytes / 2, tU, full, x, y);
    ++loads;
  };
  int fc = 0, y = 0, nfc = 0, ny = 0;
  int t = next_valid((int)blockIdx.x / 2, fc, y);
  if (t < nt) load(fc, y);
  bool ok = true;
  for (uint32_t g = 0; ok && t < nt; g += 4) {
    const int tn = next_valid(t + step, nfc, ny);
    for (int c = 0; c < 4; ++c) {
      if (!mbar_wait(written, (g + (uint32_t)c) & 1u, &s.abort, p.err)) { ok = false; break; }
      tma_store_2d(tO0, set, fc + 32 * c, y);
      tma_store_2d(tO1, set + kMxHuSetBytes / 2, fc + 32 * c, y);
      tma_store_2d(tQ0, cbuf, fc + 32 * c, y);
      tma_store_2d(tQ1, cbuf + kTileM * 32, fc + 32 * c, y);
      bulk_commit();
      bulk_wait_read_all();
      mbar_arrive(&s.codefree[half]);
      // the set's next chunk: c + 1 of this tile, else chunk 0 of the next tile
      if (c + 1 < 4) load(fc + 32 * (c + 1), y);
      else if (tn < nt) load(nfc, ny);
    }
    t = tn;
    fc = nfc;
    y = ny;
  }
  if (!ok && loads > 0) {   // the last copy into the set may still be in flight: let it land
    const uint32_t a = smem_u32(full);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(a, (loads - 1u) & 1u) && globaltimer() - t0 < 100000ull) {}
  }
  bulk_wait_all();   // stores complete before the CTA exits
}

__global__ void __launch_bounds__(kMxPairThreads, 1)
    grouped_gemm_mx_pair_kernel(const __grid_constant__ CUtensorMap tA0,
                                const __grid_constant__ CUtensorMap tA1,
                                const __grid_constant__ CUtensorMap tB0,
                                const __grid_constant__ CUtensorMap tB1,
                                const __grid_constant__ CUtensorMap tSA0,
                                const __grid_constant__ CUtensorMap tSA1,
                                const __grid_constant__ CUtensorMap tSB0,
                                const __grid_constant__ CUtensorMap tSB1,
                                const __grid_constant__ CUtensorMap tO0,
                                const __grid_constant__ CUtensorMap tO1,
                                const __grid_constant__ CUtensorMap tH,
                                const __grid_constant__ CUtensorMap tU,
                                const __grid_constant__ CUtensorMap tQ0,
                                const __grid_constant__ CUtensorMap tQ1, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    pdl_wait();
    if (threadIdx.x == 0) raise_error(p.err, MOE_DEVERR_BOUNDS);
    return;
  }
  uint8_t* ring = smem_raw;
  Ctl& s = *reinterpret_cast<Ctl*>(smem_raw + kRingBytes + 2 * kStageOutBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.tfull[0], 1);
    mbar_init(&s.tempty[0], 2 * kEpiThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.hufull[i], 1);
      mbar_init(&s.huwritten[i], kEpiThreads / 2);
      mbar_init(&s.codefree[i], 1);
    }
    mbar_init(&s.fin, 1);
    s.abort = 0;
    fence_barrier_init();
  }
  pdl_wait();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s.tile_off[i] = p.tile_offsets[i];
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < p.E; ++e) {
      s.pair_off[e] = run;
      run += (s.tile_off[e + 1] - s.tile_off[e] + 1) / 2;
    }
    s.pair_off[p.E] = run;
  }
  cluster_sync();   // both CTAs' barriers are initialised before any remote arrive
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tA0);
    prefetch_tensormap(&tA1);
    prefetch_tensormap(&tB0);
    prefetch_tensormap(&tB1);
    prefetch_tensormap(&tSA0);
    prefetch_tensormap(&tSA1);
    prefetch_tensormap(&tSB0);
    prefetch_tensormap(&tSB1);
    prefetch_tensormap(&tO0);
    prefetch_tensormap(&tO1);
    if (p.epi == EPI_SWIGLU_BWD_MX) {
      prefetch_tensormap(&tH);
      prefetch_tensormap(&tU);
      prefetch_tensormap(&tQ0);
      prefetch_tensormap(&tQ1);
    }
  }
  if (warp == 1) tmem_alloc_pair(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s.tmem_base;

  if (warp < 4) {
    setmaxnreg_dec<kMxPairRoleRegs>();
    if (warp == 0 && lane == 0) {
      const MxMaps mp = {{&tA0, &tA1}, {&tB0, &tB1}, {&tSA0, &tSA1}, {&tSB0, &tSB1}};
      producer_mx_pair(p, s, ring, rank, mp);
    } else if (warp == 1 && lane == 0) {
      mma_issuer_mx_pair(p, s, ring, tmem_base, rank);
    } else if (warp >= 2 && lane == 0 && p.epi == EPI_SWIGLU_BWD_MX) {
      hu_mover_mx_pair(p, s, rank, warp - 2, ring + p.stages * p.stage_bytes, &tO0, &tO1, &tH,
                       &tU, &tQ0, &tQ1);
    }
  } else {
    setmaxnreg_inc<kMxPairEpiRegs>();
    epilogue_mx_pair(p, s, tmem_base, warp, lane, rank, ring + p.stages * p.stage_bytes, &tO0,
                     &tO1, &tQ0, &tQ1);
  }

  tc_fence_before();
  cluster_sync();   // the partner no longer reads this CTA's memory
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
std::atomic<int> g_inject_stall{0};

// The bf16 data GEMMs run on CTA pairs (measured on the 8192-token, 32-expert
// layer against single CTAs: fwd2 -6%, dgrad1 -8%, wgrad2 -11%, wgrad1 -13%,
// fwd1 -3%, dgrad2 -4%); the narrow router GEMM stays on single CTAs.
bool op_uses_pairs(int op) {
  return op == OP_FWD1_SWIGLU || op == OP_FWD2 || op == OP_DGRAD2_SWIGLU || op == OP_DGRAD1 ||
         op == OP_WGRAD1 || op == OP_WGRAD2 || op == OP_WGRAD1_NAT || op == OP_WGRAD2_NAT;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// box of box_inner x box_outer, 128-byte swizzle, zero fill out of bounds.
enum MapType { MAP_BF16 = 0, MAP_U8 = 1, MAP_F32 = 2 };
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, int type = MAP_BF16, int swizzle = 128) {
  const int esz = type == MAP_U8 ? 1 : (type == MAP_F32 ? 4 : 2);
  const CUtensorMapDataType dt = type == MAP_U8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : (type == MAP_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                    : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle == 32    ? CU_TENSOR_MAP_SWIZZLE_32B
                  : swizzle == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                  : swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte view of an MXFP8 scale array (sf_offset layout) of a K-major
// [rows, K] operand: two 256-byte rows per 512-byte atom, one atom per box.
bool make_sf_map(CUtensorMap* m, const void* sf, uint64_t rows, uint64_t K) {
  return make_map(m, sf, 256, rows / kTileM * (K / 128) * 2, 256, 2, MAP_U8, 0);
}

// Pairs that can be resident at once (the persistent grid of the pair kernels,
// which all have the same shared memory and threads per CTA).
int resident_pairs(const DeviceInfo* di) {
  static int resident[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return di->sm_count / 2;
  if (resident[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)di->sm_count);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<false, true>, &cfg) != cudaSuccess ||
        n < 1)
      n = di->sm_count / 2;
    resident[dev] = n;
  }
  return resident[dev];
}

// MXFP8 data GEMM on CTA pairs: `p` arrives set up for 128-column tiles (maps
// with 128 x 128-code boxes, n_tiles of 128); N is a multiple of 256.
cudaError_t launch_mx_pair(Params p, const CUtensorMap& A0, const CUtensorMap& A1,
                           const CUtensorMap& B0, const CUtensorMap& B1, const GemmLaunch& g,
                           const DeviceInfo* di, cudaStream_t stream) {
  const uint64_t rows = (uint64_t)g.rows_max;
  p.n_tiles = p.n_tiles * p.BN / kMxPairBN;
  p.BN = kMxPairBN;
  p.kstep = 128;
  p.acc_cols = 256;
  p.num_acc = 1;
  p.tmem_cols = (int)kTmemCols;
  p.stages = p.epi == EPI_SWIGLU_BWD_MX ? kMxBwdStages : kMxPairStages;
  p.stage_bytes = kMxPairStageBytes;
  p.tx_bytes = kMxPairTx;
  p.tma_store = 0;
  const uint64_t ka = (uint64_t)p.sf_ka * 128, kb = (uint64_t)p.sf_kb * 128;
  const uint64_t brows = (uint64_t)g.E * (uint64_t)p.b_group_rows;
  CUtensorMap SA0, SA1, SB0, SB1;
  bool ok = make_sf_map(&SA0, p.sfa0, rows, ka) && make_sf_map(&SB0, p.sfb0, brows, kb);
  SA1 = SA0;
  SB1 = SB0;
  if (ok && p.sfa1 != p.sfa0) ok = make_sf_map(&SA1, p.sfa1, rows, ka);
  if (ok && p.sfb1 != p.sfb0) ok = make_sf_map(&SB1, p.sfb1, brows, kb);
  // bf16 outputs: out0 (H, Y, dH or dXd) and out1 (U or dU), 32-column boxes
  CUtensorMap O0, O1;
  const uint64_t ocols = (uint64_t)p.ldo;
  ok = ok && make_map(&O0, p.out0, ocols, rows, 32, kTileM, MAP_BF16, 64);
  O1 = O0;
  if (ok && p.out1 != nullptr) ok = make_map(&O1, p.out1, ocols, rows, 32, kTileM, MAP_BF16, 64);
  // SwiGLU backward: H (aux0) and U (aux1) in the same 32-column boxes
  // and the E4M3 codes of dH (out2) and dU (out3): 32-byte boxes, 32-byte swizzle
  CUtensorMap MH = O0, MU = O0, QH = O0, QU = O0;
  if (ok && p.epi == EPI_SWIGLU_BWD_MX)
    ok = make_map(&MH, p.aux0, ocols, rows, 32, kTileM, MAP_BF16, 64) &&
         make_map(&MU, p.aux1, ocols, rows, 32, kTileM, MAP_BF16, 64) &&
         make_map(&QH, p.out2, ocols, rows, 32, kTileM, MAP_U8, 32) &&
         make_map(&QU, p.out3, ocols, rows, 32, kTileM, MAP_U8, 32);
  // SwiGLU forward: A's codes (out2, 64-byte boxes) and, when asked for, A
  // dequantised (out3, bf16, 32-column boxes), both with the 64-byte swizzle
  if (ok && p.epi == EPI_SWIGLU_FWD_MX) {
    ok = make_map(&QU, p.out2, ocols, rows, 64, kTileM, MAP_U8, 64);
    if (ok && p.out3 != nullptr) ok = make_map(&QH, p.out3, ocols, rows, 32, kTileM, MAP_BF16, 64);
  }
  if (!ok) return cudaErrorInvalidValue;
  // the register split above assumes the launch allocation it was computed for
  // (a smaller one would leave setmaxnreg.inc waiting for registers forever)
  static int launch_regs = -1;
  if (launch_regs < 0) {
    cudaFuncAttributes fa = {};
    launch_regs = cudaFuncGetAttributes(&fa, grouped_gemm_mx_pair_kernel) == cudaSuccess ? fa.numRegs : 0;
  }
  if (launch_regs != kMxPairLaunchRegs) return cudaErrorInvalidConfiguration;
  const int64_t pairs = ((int64_t)(rows / kTileM) / 2 + g.E) * p.n_tiles;
  int64_t np = resident_pairs(di);
  if (pairs < np) np = pairs;
  if (np < 1) np = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * np));
  cfg.blockDim = dim3(kMxPairThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_mx_pair_kernel, A0, A1, B0, B1, SA0, SA1, SB0, SB1,
                            O0, O1, MH, MU, QH, QU, p);
}

}  // namespace

int gemm_set_inject_stall(int mode) { return g_inject_stall.exchange(mode); }

cudaError_t gemm_init_attributes() {
  if (!get_encoder()) return cudaErrorInitializationError;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<false, true, false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_kernel<false, true, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_mx_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_grouped_gemm(const GemmLaunch& g, cudaStream_t stream) {
  if (!get_encoder()) return cudaErrorInitializationError;
  const DeviceInfo* di = device_info();
  if (di == nullptr || !di->ready) return cudaErrorInitializationError;
  Params p = {};
  CUtensorMap A0, A1, B0, B1, O0, O1, O2;
  const uint64_t rows = (uint64_t)g.rows_max;
  const int d = g.d, f = g.f, E = g.E;
  bool ok = true;
  p.E = E;
  p.tile_offsets = g.tile_offsets;
  p.rows_max = g.rows_max;
  p.err = g.err;
  p.k_split = 1 << 30;
  p.m_split = 1 << 30;
  p.k_parts = 1;
  p.kstep = kBK;
  p.acc_cols = 256;
  p.inject_stall = g_inject_stall.load();
  p.num_acc = 2;
  p.tmem_cols = (int)kTmemCols;
  bool mx = false;
  int64_t max_tiles = 0;
  switch (g.op) {
    case OP_FWD1_SWIGLU:
      p.mode = MODE_MGROUP; p.epi = EPI_SWIGLU_FWD; p.b_dual = 1; p.BN = 256;
      p.n_tiles = f / 128; p.k_steps = d / kBK; p.b_group_rows = f;
      ok = make_map(&A0, g.a0, d, rows, 64, 128) && make_map(&B0, g.w0, d, (uint64_t)E * f, 64, 128) &&
           make_map(&B1, g.w1, d, (uint64_t)E * f, 64, 128);
      A1 = A0;
      p.out0 = g.out0; p.out1 = g.out1; p.out2 = g.out2; p.ldo = f;
      ok = ok && make_map(&O0, g.out0, f, rows, 64, 128) && make_map(&O1, g.out1, f, rows, 64, 128) &&
           make_map(&O2, g.out2, f, rows, 64, 128);
      p.tma_store = 1;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_FWD2:
      p.mode = MODE_MGROUP; p.epi = EPI_BF16; p.BN = (d % 256 == 0) ? 256 : 128;
      p.n_tiles = d / p.BN; p.k_steps = f / kBK; p.b_group_rows = d;
      ok = make_map(&A0, g.a0, f, rows, 64, 128) &&
           make_map(&B0, g.w0, f, (uint64_t)E * d, 64, (uint32_t)p.BN);
      A1 = A0; B1 = B0;
      p.out0 = g.out0; p.ldo = d;
      ok = ok && make_map(&O0, g.out0, d, rows, 64, 128);
      O1 = O2 = O0;
      p.tma_store = 1;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_DGRAD2_SWIGLU:
      p.mode = MODE_MGROUP; p.epi = EPI_SWIGLU_BWD; p.b_mn = 1; p.BN = (f % 256 == 0) ? 256 : 128;
      p.n_tiles = f / p.BN; p.k_steps = d / kBK; p.b_group_rows = d;
      ok = make_map(&A0, g.a0, d, rows, 64, 128) && make_map(&B0, g.w0, f, (uint64_t)E * d, 64, 64);
      A1 = A0; B1 = B0;
      p.out0 = g.out0; p.out1 = g.out1; p.aux0 = g.aux0; p.aux1 = g.aux1; p.ldo = f;
      ok = ok && make_map(&O0, g.out0, f, rows, 32, 128, MAP_BF16, 64) &&
           make_map(&O1, g.out1, f, rows, 32, 128, MAP_BF16, 64);
      O2 = O0;
      p.tma_store = 1;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_DGRAD1:
      p.mode = MODE_MGROUP; p.epi = EPI_BF16; p.b_mn = 1; p.BN = (d % 256 == 0) ? 256 : 128;
      p.n_tiles = d / p.BN; p.k_steps = 2 * f / kBK; p.k_split = f / kBK; p.b_group_rows = f;
      ok = make_map(&A0, g.a0, f, rows, 64, 128) && make_map(&A1, g.a1, f, rows, 64, 128) &&
           make_map(&B0, g.w0, d, (uint64_t)E * f, 64, 64) &&
           make_map(&B1, g.w1, d, (uint64_t)E * f, 64, 64);
      p.out0 = g.out0; p.ldo = d;
      ok = ok && make_map(&O0, g.out0, d, rows, 64, 128);
      O1 = O2 = O0;
      p.tma_store = 1;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_WGRAD2:
      p.mode = MODE_KGROUP; p.epi = EPI_F32; p.a_mn = 1; p.b_mn = 1;
      p.BN = (f % 256 == 0) ? 256 : 128; p.m_tiles = d / kTileM; p.n_tiles = f / p.BN;
      ok = make_map(&A0, g.a0, d, rows, 64, 64) && make_map(&B0, g.a1, f, rows, 64, 64);
      A1 = A0; B1 = B0;
      p.out0 = g.out0; p.ldo = f; p.out_group_stride = (int64_t)d * f;
      ok = ok && make_map(&O0, g.out0, f, (uint64_t)E * d, 32, 128, MAP_F32);
      O1 = O2 = O0;
      p.tma_store = 1;
      p.out_rows_per_group = d;
      max_tiles = (int64_t)E * p.m_tiles * p.n_tiles;
      break;
    case OP_WGRAD1:
      p.mode = MODE_KGROUP; p.epi = EPI_F32; p.a_mn = 1; p.b_mn = 1;
      p.BN = (d % 256 == 0) ? 256 : 128; p.m_tiles = 2 * f / kTileM; p.m_split = f / kTileM;
      p.n_tiles = d / p.BN;
      ok = make_map(&A0, g.a0, f, rows, 64, 64) && make_map(&A1, g.a1, f, rows, 64, 64) &&
           make_map(&B0, g.aux0, d, rows, 64, 64);
      B1 = B0;
      p.out0 = g.out0; p.out1 = g.out1; p.ldo = d; p.out_group_stride = (int64_t)f * d;
      ok = ok && make_map(&O0, g.out0, d, (uint64_t)E * f, 32, 128, MAP_F32) &&
           make_map(&O1, g.out1, d, (uint64_t)E * f, 32, 128, MAP_F32);
      O2 = O0;
      p.tma_store = 1;
      p.out_rows_per_group = f;
      max_tiles = (int64_t)E * p.m_tiles * p.n_tiles;
      break;
    case OP_WGRAD2_NAT:   // B = A_q (codes [rows, f]) dequantised in the kernel
      if (!natural_wgrad_supported(g.op, d, f)) return cudaErrorInvalidValue;
      p.mode = MODE_KGROUP; p.epi = EPI_F32; p.a_mn = 1; p.b_mn = 1; p.dq_b = 1;
      p.BN = 256; p.m_tiles = d / kTileM; p.n_tiles = f / p.BN;
      ok = make_map(&A0, g.a0, d, rows, 64, 64) && make_map(&B0, g.a1, f, rows, 128, kBK, MAP_U8, 0);
      A1 = A0; B1 = B0;
      p.sfq = g.sfb0; p.sfq_k = f / 128;
      p.out0 = g.out0; p.ldo = f; p.out_group_stride = (int64_t)d * f;
      ok = ok && make_map(&O0, g.out0, f, (uint64_t)E * d, 32, 128, MAP_F32);
      O1 = O2 = O0;
      p.tma_store = 1;
      p.out_rows_per_group = d;
      max_tiles = (int64_t)E * p.m_tiles * p.n_tiles;
      break;
    case OP_WGRAD1_NAT:   // B = Xd_q (codes [rows, d]) dequantised in the kernel
      if (!natural_wgrad_supported(g.op, d, f)) return cudaErrorInvalidValue;
      p.mode = MODE_KGROUP; p.epi = EPI_F32; p.a_mn = 1; p.b_mn = 1; p.dq_b = 1;
      p.BN = 256; p.m_tiles = 2 * f / kTileM; p.m_split = f / kTileM;
      p.n_tiles = d / p.BN;
      ok = make_map(&A0, g.a0, f, rows, 64, 64) && make_map(&A1, g.a1, f, rows, 64, 64) &&
           make_map(&B0, g.aux0, d, rows, 128, kBK, MAP_U8, 0);
      B1 = B0;
      p.sfq = g.sfb0; p.sfq_k = d / 128;
      p.out0 = g.out0; p.out1 = g.out1; p.ldo = d; p.out_group_stride = (int64_t)f * d;
      ok = ok && make_map(&O0, g.out0, d, (uint64_t)E * f, 32, 128, MAP_F32) &&
           make_map(&O1, g.out1, d, (uint64_t)E * f, 32, 128, MAP_F32);
      O2 = O0;
      p.tma_store = 1;
      p.out_rows_per_group = f;
      max_tiles = (int64_t)E * p.m_tiles * p.n_tiles;
      break;
    case OP_ROUTER: {
      p.mode = MODE_DENSE; p.epi = EPI_ROUTER; p.BN = ((E + 15) / 16) * 16;
      p.n_tiles = 1; p.m_tiles = (g.T + kTileM - 1) / kTileM; p.m_valid = g.T; p.n_valid = E;
      p.k_steps = d / kBK;
      ok = make_map(&A0, g.a0, d, (uint64_t)g.T, 64, 128) &&
           make_map(&B0, g.w0, d, (uint64_t)E, 64, (uint32_t)p.BN);
      A1 = A0; B1 = B0;
      p.out0 = g.out0; p.bias = g.bias;
      // few row tiles: two CTAs per tile, each over half of K (the logits are
      // zeroed first and both halves are added atomically)
      if (2 * p.m_tiles <= di->sm_count && p.k_steps % 2 == 0) {
        p.k_parts = 2;
        if (cudaMemsetAsync(g.out0, 0, (size_t)g.T * E * sizeof(float), stream) != cudaSuccess)
          return cudaErrorInvalidValue;
      }
      max_tiles = (int64_t)p.m_tiles * p.k_parts;
      break;
    }
    // ---- MXFP8: 128x128 tiles, K steps of 128 fp8 (128 bytes), scales per stage
    case OP_MX_FWD1_SWIGLU:
      mx = true; p.mode = MODE_MGROUP; p.epi = EPI_SWIGLU_FWD_MX; p.BN = 128;
      p.n_tiles = 2 * f / 128; p.k_steps = d / 128; p.b_group_rows = 2 * f;
      ok = make_map(&A0, g.a0, d, rows, 128, 128, MAP_U8) &&
           make_map(&B0, g.w0, d, (uint64_t)E * 2 * f, 128, 128, MAP_U8);
      A1 = A0; B1 = B0;
      p.sfa0 = p.sfa1 = g.sfa0; p.sfb0 = p.sfb1 = g.sfb0; p.sf_ka = p.sf_kb = d / 128;
      p.out0 = g.out0; p.out1 = g.out1; p.out2 = g.out2; p.out3 = g.out3; p.osf0 = g.osf0;
      p.osf_kb = f / 32;
      p.ldo = f;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_MX_FWD2:
      mx = true; p.mode = MODE_MGROUP; p.epi = EPI_BF16; p.BN = 128;
      p.n_tiles = d / 128; p.k_steps = f / 128; p.b_group_rows = d;
      ok = make_map(&A0, g.a0, f, rows, 128, 128, MAP_U8) &&
           make_map(&B0, g.w0, f, (uint64_t)E * d, 128, 128, MAP_U8);
      A1 = A0; B1 = B0;
      p.sfa0 = p.sfa1 = g.sfa0; p.sfb0 = p.sfb1 = g.sfb0; p.sf_ka = p.sf_kb = f / 128;
      p.out0 = g.out0; p.ldo = d;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_MX_DGRAD2_SWIGLU:
      mx = true; p.mode = MODE_MGROUP; p.epi = EPI_SWIGLU_BWD_MX; p.BN = 128;
      p.n_tiles = f / 128; p.k_steps = d / 128; p.b_group_rows = f;
      ok = make_map(&A0, g.a0, d, rows, 128, 128, MAP_U8) &&
           make_map(&B0, g.w0, d, (uint64_t)E * f, 128, 128, MAP_U8);
      A1 = A0; B1 = B0;
      p.sfa0 = p.sfa1 = g.sfa0; p.sfb0 = p.sfb1 = g.sfb0; p.sf_ka = p.sf_kb = d / 128;
      p.aux0 = g.aux0; p.aux1 = g.aux1;
      p.out0 = g.out0; p.out1 = g.out1; p.out2 = g.out2; p.out3 = g.out3;
      p.osf0 = g.osf0; p.osf1 = g.osf1; p.osf_kb = f / 32; p.ldo = f;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    case OP_MX_DGRAD1:
      mx = true; p.mode = MODE_MGROUP; p.epi = EPI_BF16; p.BN = 128;
      p.n_tiles = d / 128; p.k_steps = 2 * f / 128; p.k_split = f / 128; p.b_group_rows = d;
      ok = make_map(&A0, g.a0, f, rows, 128, 128, MAP_U8) && make_map(&A1, g.a1, f, rows, 128, 128, MAP_U8) &&
           make_map(&B0, g.w0, f, (uint64_t)E * d, 128, 128, MAP_U8) &&
           make_map(&B1, g.w1, f, (uint64_t)E * d, 128, 128, MAP_U8);
      p.sfa0 = g.sfa0; p.sfa1 = g.sfa1; p.sfb0 = g.sfb0; p.sfb1 = g.sfb1; p.sf_ka = p.sf_kb = f / 128;
      p.out0 = g.out0; p.ldo = d;
      max_tiles = (int64_t)(rows / kTileM) * p.n_tiles;
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (!ok) return cudaErrorInvalidValue;
  if (mx && (p.n_tiles * p.BN) % kMxPairBN == 0)
    return launch_mx_pair(p, A0, A1, B0, B1, g, di, stream);
  if (!p.tma_store) O0 = O1 = O2 = A0;   // unused by the direct-store epilogues
  // CTA pairs: bf16 M-grouped GEMMs, and K-grouped ones with an even number of M tiles
  const bool pair = op_uses_pairs(g.op) && !mx && p.tma_store &&
                    (p.mode == MODE_MGROUP || (p.mode == MODE_KGROUP && p.m_tiles % 2 == 0));
  if (p.dq_b && !pair) return cudaErrorInvalidValue;
  if (pair && p.BN == 128 && g.op != OP_FWD1_SWIGLU) {
    // N = 128 (mod 256): 256-wide pair tiles (half the operand bytes per flop
    // of 128-wide ones), the last tile running 128 columns past N
    const int n_cols = p.n_tiles * 128;
    max_tiles = max_tiles / p.n_tiles * ((n_cols + 255) / 256);
    p.BN = 256;
    p.n_tiles = (n_cols + 255) / 256;
    p.n_cols = n_cols;
  }
  if (pair && p.mode == MODE_MGROUP && !p.b_mn && !p.b_dual) {
    // K-major B: each CTA of the pair loads BN/2 rows
    const void* wb = (g.op == OP_FWD2) ? g.w0 : nullptr;
    if (wb == nullptr || !make_map(&B0, wb, f, (uint64_t)E * d, 64, (uint32_t)(p.BN / 2)))
      return cudaErrorInvalidValue;
    B1 = B0;
  }
  if (mx) {
    p.kstep = 128;
    p.acc_cols = 128;
    p.tx_bytes = kABytes + p.BN * 128 + 512 * (1 + p.BN / 128);
    p.stage_bytes = (p.tx_bytes + 1023) & ~1023;
  } else if (p.dq_b) {
    // the ring holds A + codes + scale atom per stage; B's bf16 slots follow it
    p.pair_half_bytes = kABytes;
    p.tx_bytes = 2 * kABytes;
    p.stage_bytes = kDqStageBytes;
    p.num_acc = 2;
    p.tmem_cols = 512;
  } else if (pair) {
    p.pair_half_bytes = kABytes + (p.BN / 2) * kBK * 2;
    p.tx_bytes = 2 * p.pair_half_bytes;
    p.stage_bytes = p.pair_half_bytes;
    // two 256-column accumulators per CTA: the pair's allocation is collective
    // (both CTAs receive the same columns)
    p.num_acc = 2;
    p.tmem_cols = 512;
  } else {
    p.tx_bytes = kABytes + (p.b_dual ? kBBytesMax : p.BN * kBK * 2);
    p.stage_bytes = p.tx_bytes;
  }
  p.stages = p.dq_b ? kDqStages : kRingBytes / p.stage_bytes;
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  if (p.stages < 2 || p.stage_bytes % 1024 != 0) return cudaErrorInvalidValue;
  int grid = (int)(max_tiles < di->sm_count ? max_tiles : di->sm_count);
  if (grid < 1) grid = 1;
  if (pair) {
    const int64_t pairs = (p.mode == MODE_MGROUP) ? (max_tiles / 2 + (int64_t)E * p.n_tiles)
                                                  : max_tiles / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(p.dq_b ? kThreadsDq : kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many pairs as can be resident at once (persistent tile loop)
    int64_t np = resident_pairs(di);
    if (pairs < np) np = pairs;
    if (np < 1) np = 1;
    cfg.gridDim = dim3((unsigned)(2 * np));
    cudaLaunchAttribute attr2[2] = {attr[0], {}};
    attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr2[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr2;
    cfg.numAttrs = 2;
    // (the dequantising kernel has the same shared memory: one CTA per SM too)
    if (p.dq_b)
      return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false, true, true>, A0, A1, B0, B1, O0,
                                O1, O2, p);
    if (p.mode == MODE_KGROUP)
      return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false, true, false, true>, A0, A1, B0, B1,
                                O0, O1, O2, p);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false, true>, A0, A1, B0, B1, O0, O1, O2,
                              p);
  }
  if (mx)
    return launch_pdl(grouped_gemm_kernel<true, false>, dim3(grid), dim3(kThreads), kSmemBytes,
                      stream, A0, A1, B0, B1, O0, O1, O2, p);
  return launch_pdl(grouped_gemm_kernel<false, false>, dim3(grid), dim3(kThreads), kSmemBytes,
                    stream, A0, A1, B0, B1, O0, O1, O2, p);
}

MOE_CHECK_WORD_ACCESSOR(gemm)

}  // namespace moe
