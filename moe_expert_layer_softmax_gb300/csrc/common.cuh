// Shared device helpers for the sm_103a MoE layer kernels: bf16 packing,
// error word, mbarrier / TMA / tcgen05 wrappers (inline PTX) and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

constexpr int kTileM = MOE_TILE_M;   // grouped-GEMM tile rows == expert padding unit
constexpr int kWarp = 32;

// A bounded on-chip wait gives up after this many nanoseconds of %globaltimer.
// Healthy waits in these kernels last microseconds; a second means a lost arrive.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

// ------------------------------------------------------------------ bf16
MOE_DEV float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
MOE_DEV void unpack8(const uint4& v, float* f) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}
MOE_DEV uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                    pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

MOE_DEV void raise_error(int32_t* err, int bits) {
  if (err != nullptr) atomicOr(err, bits);
}

// ---------------------------------------------------------------- checks build
// Built with -DMOE_CHECKS (a test build that stands in for a memory checker),
// every index that a kernel reads from device data (a slot, a route, a padding
// row, a tile's rows) is checked against its buffer before the access it
// guards: an index outside sets MOE_DEVERR_BOUNDS in the translation unit's
// check word (moe_checks_read() collects them) and the access is skipped.  The
// normal build compiles none of this: MOE_CHECKED(i, n) { ... } is then a
// plain block.
#ifdef MOE_CHECKS
static __device__ int32_t g_check_word;
MOE_DEV bool checked_index(int64_t i, int64_t n) {
  const bool ok = i >= 0 && i < n;
  if (!ok) atomicOr(&g_check_word, MOE_DEVERR_BOUNDS);
  return ok;
}
#define MOE_CHECKED(i, n) if (::moe::checked_index((int64_t)(i), (int64_t)(n)))
#define MOE_CHECK_OK(i, n) ::moe::checked_index((int64_t)(i), (int64_t)(n))
// host side: this translation unit's check word (device address), or NULL
#define MOE_CHECK_WORD_ACCESSOR(name)                                                  \
  int32_t* check_word_##name() {                                                       \
    void* p = nullptr;                                                                 \
    return cudaGetSymbolAddress(&p, g_check_word) == cudaSuccess ? static_cast<int32_t*>(p) \
                                                                 : nullptr;            \
  }
#else
#define MOE_CHECKED(i, n)
#define MOE_CHECK_OK(i, n) true
#define MOE_CHECK_WORD_ACCESSOR(name) \
  int32_t* check_word_##name() { return nullptr; }
#endif

// rows of the dispatched buffers: T*k + E*(MOE_TILE_M-1), rounded up to a tile
MOE_DEV int64_t rows_max_of(int T, int k, int E) {
  return ((int64_t)T * k + (int64_t)E * (MOE_TILE_M - 1) + MOE_TILE_M - 1) / MOE_TILE_M * MOE_TILE_M;
}

MOE_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
MOE_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase of `bar` with the given parity has completed.  Gives up
// (returns false) when *abort is set by another role or after kWaitLimitNs; on
// a timeout it sets *abort and the TIMEOUT bit of the error word.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 127u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        raise_error(err, MOE_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ TMA
MOE_DEV void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation (launch_pdl): it may be scheduled
// while the previous kernel of the stream is still finishing.  Each kernel
// first allows its own successor to be scheduled, then calls pdl_wait()
// before its first global-memory access: pdl_wait() returns once the
// previous kernel has completed and its writes are visible.
MOE_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
MOE_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void pdl_begin() {
  pdl_launch_dependents();
  pdl_wait();
}

MOE_DEV void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// TMA store of a 2-D box from shared memory (bulk-group completion).
MOE_DEV void tma_store_2d(const CUtensorMap* map, const void* smem_src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y)
      : "memory");
}
MOE_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has read its source.
MOE_DEV void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store of this thread has completed.
MOE_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's shared-memory writes visible to the async (TMA) proxy.
MOE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier over `n` threads.
MOE_DEV void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Named barrier that also returns the AND of every participant's `v`.
MOE_DEV bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ tcgen05
// Shared-memory matrix descriptor, 128-byte swizzle (descriptor version 1).
//   K-major tiles: rows of 128 B (64 bf16 along K), 8-row groups 1024 B apart
//                  (stride byte offset); the leading offset is unused.
//   MN-major tiles: rows of 128 B (64 bf16 along M/N) indexed by K, 8-row groups
//                  1024 B apart (stride byte offset), 64-element M/N blocks
//                  `lbo` bytes apart (leading byte offset).
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
MOE_DEV uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;                       // D format: f32
  d |= 1u << 7;                       // A format: bf16
  d |= 1u << 10;                      // B format: bf16
  d |= (uint32_t)(a_mn_major & 1) << 15;
  d |= (uint32_t)(b_mn_major & 1) << 16;
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

MOE_DEV void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Block-scaled MXFP8 MMA (E4M3 x E4M3, E8M0 scales in tensor memory, one
// scale per 32 K-values; the scale byte of this K=32 step is chosen by the
// scale-factor ids in the instruction descriptor).
MOE_DEV void tc_mma_mxf8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t tmem_sfa, uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(tmem_sfa), "r"(tmem_sfb)
      : "memory");
}

// Instruction descriptor for kind::mxf8f6f4 with E4M3 A/B, UE8M0 scales,
// fp32 accumulation, K-major operands; sf_id picks the scale byte.
MOE_DEV uint32_t idesc_mxf8(int M, int N, int sf_id) {
  uint32_t d = 0;
  d |= (uint32_t)(sf_id & 3) << 4;    // B scale-factor byte
  d |= (uint32_t)(N >> 3) << 17;
  d |= 1u << 23;                      // scale type: UE8M0
  d |= (uint32_t)(M >> 4) << 24;
  d |= (uint32_t)(sf_id & 3) << 29;   // A scale-factor byte
  return d;
}

// Copy 32 rows x 16 bytes of shared memory into tensor-memory lanes 0-31 and
// replicate them to the other three lane quarters.
MOE_DEV void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Shared-memory descriptor without swizzle: 16-byte rows, 8-row groups 128 B apart.
MOE_DEV uint64_t smem_desc_noswz(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Plain bulk copy global -> shared, completion counted on `bar`.
MOE_DEV void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
MOE_DEV void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Warp-wide: allocate `ncols` TMEM columns, base address written to *dst (smem).
MOE_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets row
// (lane base + i), columns [col, col + 32).  The wait for the load is part of
// the same asm statement, so the registers are valid when it returns.
MOE_DEV void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Two such loads (e.g. the gate and up halves of a SwiGLU tile) and one wait.
MOE_DEV void tmem_ld32x2(uint32_t taddr0, uint32_t taddr1, uint32_t* r, uint32_t* q) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]), "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]), "=r"(q[14]), "=r"(q[15]), "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]), "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]), "=r"(q[25]), "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
}

// ------------------------------------------------------------------ CTA pairs
// (clusters of two CTAs sharing one tcgen05 MMA of M = 256)
MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
MOE_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// every thread of both CTAs
MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address)
MOE_DEV void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t mbar_cluster, int x,
                              int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster), "r"(x), "r"(y)
      : "memory");
}
// Arrive on an mbarrier of either CTA of the pair.  The release is at CTA
// scope (the usual form for tcgen05 pipelines: what the arriving threads hand
// over is read by tensor-core operations, ordered by the proxy and tcgen05
// fences before the arrive); a cluster-scope release adds a memory barrier per
// arrive that measured about 1 us under load, on the critical path of a
// per-stage hand-off.
MOE_DEV void mbar_arrive_cluster(uint32_t mbar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(mbar_cluster)
               : "memory");
}
MOE_DEV void tc_mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Block-scaled MXFP8 MMA of a CTA pair (M = 256): each CTA reads its own A
// rows from its shared memory and its A scales from its own tensor memory;
// the B scales of all N columns must be present in both CTAs' tensor memory.
MOE_DEV void tc_mma_mxf8_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t tmem_sfa, uint32_t tmem_sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(tmem_sfa), "r"(tmem_sfb)
      : "memory");
}
// Pair form of tc_cp_32x128b_x4, issued by the even CTA: each CTA's copy of the
// 32 x 16-byte block at this shared-memory offset goes to its own tensor memory.
MOE_DEV void tc_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Warpgroup-wide register reallocation (every warp of the warpgroup executes it).
template <int N>
MOE_DEV void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
MOE_DEV void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// arrive once on the mbarrier at this offset in both CTAs of the pair when all
// tcgen05 operations issued so far by this thread have completed
MOE_DEV void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
// warp-wide, in both CTAs: the pair's tensor memory (same columns in each CTA)
MOE_DEV void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc_pair(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols)
               : "memory");
}

// ------------------------------------------------------------------ MXFP8
// One E8M0 scale per 32 consecutive values along the contraction axis:
// 2^s with s the smallest integer such that amax <= 448 * 2^s, clamped to
// [-127, 127] (s = 0 for an all-zero block); codes are E4M3(v / 2^s), round
// to nearest even, saturating.  From the bits of amax = 1.m * 2^(B - 127)
// (B its biased exponent) and 448 = 1.75 * 2^8: s = B - 135 when 1.m <= 1.75
// (mantissa field <= 0x600000), else B - 134.  A subnormal amax (< 2^-126)
// gives s < -127, clamped.
MOE_DEV int mx_scale_exp(float amax) {
  if (!(amax > 0.0f)) return 0;                 // zero block (a NaN never wins fmaxf)
  const uint32_t bits = __float_as_uint(amax);
  const int B = (int)(bits >> 23);              // sign bit clear
  if (B == 255) return 127;                     // infinite
  if (B == 0) return -127;
  const int s = B - ((bits & 0x7FFFFFu) <= 0x600000u ? 135 : 134);
  return s < -127 ? -127 : s;                   // B <= 254: s <= 120
}

// 2^e for e in [-127, 128], exactly (2^-127 is the subnormal with the top
// mantissa bit; 2^128 is +inf): the block scales and their inverses.
MOE_DEV float exp2i(int e) {
  return e > -127 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two floats -> two E4M3 bytes (lo in the low byte), RNE, satfinite.
MOE_DEV uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Two E4M3 bytes (low byte first) -> two floats (exact).
MOE_DEV void e4m3x2_to_f32(uint32_t two, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(two & 0xFFFFu)));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  lo = __low2float(h);
  hi = __high2float(h);
}

// Quantise 8 values (already divided by the block scale) to 8 E4M3 bytes.
MOE_DEV uint2 e4m3x8(const float* v) {
  return make_uint2(e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16),
                    e4m3x2(v[4], v[5]) | (e4m3x2(v[6], v[7]) << 16));
}

// Byte offset of the scale of (row r, K-block b) of a K-major operand with
// `kblocks` = K/32 blocks per row, in the layout the MXFP8 GEMM copies to
// tensor memory: 128-row x 4-block atoms of 512 bytes; inside an atom, row r
// and block b sit at (r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4).
MOE_DEV size_t sf_offset(int64_t r, int b, int kblocks) {
  return ((size_t)(r >> 7) * (size_t)(kblocks >> 2) + (size_t)(b >> 2)) * 512u +
         (size_t)(r & 31) * 16u + (size_t)((r & 127) >> 5) * 4u + (size_t)(b & 3);
}

}  // namespace moe
