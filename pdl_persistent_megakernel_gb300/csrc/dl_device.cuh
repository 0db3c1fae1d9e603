// dl_device.cuh -- inline-PTX building blocks for sm_103a: mbarriers, TMA
// (tiled and bulk copies), programmatic dependent launch, acquire/release
// counters, tcgen05 (TMEM allocation, MMA, commit, loads) and bounded waits.
//
// Every wait in this library is bounded by a %globaltimer budget: on expiry
// the waiting thread records DERR_TIMEOUT in the plan's status word, raises
// the abort flag and returns false; callers then drain their own copies in
// flight (again bounded), free TMEM and leave.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dl_internal.h"

namespace dl {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ trace
// Trace build: %globaltimer stamp (or a value) of share c of the current op.
__device__ __forceinline__ void trace_put(const KernelCtx& ctx, int c, int slot,
                                          unsigned long long v) {
  if (ctx.trace && c < ctx.trace_ctas)
    ctx.trace[(static_cast<size_t>(ctx.op_id) * ctx.trace_ctas + c) * kTraceSlots + slot] = v;
}
__device__ __forceinline__ void trace_stamp(const KernelCtx& ctx, int c, int slot) {
  if (ctx.trace) trace_put(ctx, c, slot, globaltimer());
}

// ------------------------------------------------------------- status word
__device__ __forceinline__ void report_error(DevStatus* st, unsigned code,
                                             unsigned op, unsigned cta,
                                             unsigned where, unsigned value) {
  if (atomicCAS(&st->code, 0u, code) == 0u) {
    st->info[0] = op;
    st->info[1] = cta;
    st->info[2] = where;
    st->info[3] = value;
    st->info[4] = blockIdx.x;
    st->info[5] = threadIdx.x;
  }
  atomicExch(&st->abort, 1u);
}

__device__ __forceinline__ bool aborted(const DevStatus* st) {
  return *reinterpret_cast<const volatile unsigned*>(&st->abort) != 0u;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// n arrivals at once (the count operand of mbarrier.arrive)
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n)
               : "memory");
}

// kCluster: acquire at cluster scope, for data that other CTAs of the
// cluster stored here with st.async completing on this barrier.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// How often a waiting thread looks at the abort flag and the budget.  The
// flag lives in global memory: reading it on every pass would make the wait
// return no sooner than one memory round trip after the phase completes,
// which under a saturated HBM is a microsecond or more.
constexpr unsigned long long kCheckNs = 20000;

// Wait for the phase with the given parity to complete; false on timeout or
// when another thread raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const KernelCtx& ctx, unsigned where) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  unsigned long long check = t0 + kCheckNs;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t = globaltimer();
    if (t >= check) {
      if (aborted(ctx.status)) return false;
      if (t - t0 > ctx.budget_ns) {
        report_error(ctx.status, DERR_TIMEOUT, ctx.op_id, blockIdx.x, where, parity);
        return false;
      }
      check = t + kCheckNs;
    }
  }
}

// Every lane of a warp waits (bounded) for the phase; the warp agrees on the
// outcome, so a timeout never splits a warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          const KernelCtx& ctx, unsigned where) {
  const bool ok = mbar_wait(bar, parity, ctx, where);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Named barrier that also ORs a predicate over the participating threads.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %3, 0;\n\t"
      "bar.red.or.pred p, %1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// Drain: wait (bounded, ignoring the abort flag) for a phase to complete.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity,
                                           unsigned long long budget_ns) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > budget_ns) return;
  }
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

// ---------------------------------------------------------- clusters
// Shared-memory address of the same variable in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Every non-exited thread of the cluster arrives (release) and waits
// (acquire); warp-uniform.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of that barrier, for a thread that arrives early and
// waits later (warp-uniform).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 4-byte store into another cluster CTA's shared memory (`addr` and `mbar`
// both from cluster_map for that CTA); it completes as 4 transaction bytes
// on that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(__float_as_uint(v)), "r"(mbar)
               : "memory");
}

// 16-byte global store with an L2 eviction-priority hint
__device__ __forceinline__ void st_global_v4_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// A descriptor that an earlier kernel wrote with ordinary stores: order
// those stores before this thread's tensor-map (TMA) reads of it.
__device__ __forceinline__ void fence_tmap_acquire(const CUtensorMap* m) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(m)
               : "memory");
}

// Prefetch one box of a tensor map into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               ::"l"(map), "r"(c0), "r"(c1) : "memory");
}

// 2-D tiled load: box at element coordinates (c0 inner, c1 outer).  c0 * the
// element size is always a multiple of 128 bytes here (one swizzle atom).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            uint64_t* bar, int c0, int c1,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_"
      "tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src,
                                          uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src),
               "r"(bytes)
               : "memory");
}

// -------------------------------------------- programmatic dependent launch
// Wait until the grids this launch depends on have completed and their
// memory is visible (no-op for launches without the PDL attribute).
__device__ __forceinline__ void gdc_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the dependent grid to be scheduled.
__device__ __forceinline__ void gdc_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------ acquire / release counters
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v)
               : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p,
                                                         unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Generic-proxy writes -> async-proxy (TMA) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Poll until *p >= value (acquire).  Bounded.
__device__ __forceinline__ bool wait_counter(const unsigned* p, unsigned value,
                                             const KernelCtx& ctx,
                                             unsigned where) {
  if (ld_acquire_gpu(p) >= value) return true;
  const unsigned long long t0 = globaltimer();
  unsigned long long check = t0 + kCheckNs;
  for (;;) {
    if (ld_acquire_gpu(p) >= value) return true;
    const unsigned long long t = globaltimer();
    if (t >= check) {
      if (aborted(ctx.status)) return false;
      if (t - t0 > ctx.budget_ns) {
        report_error(ctx.status, DERR_TIMEOUT, ctx.op_id, blockIdx.x, where, value);
        return false;
      }
      check = t + kCheckNs;
    }
  }
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          smem_u32(smem_dst)),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                   taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);       // start address
  d |= static_cast<uint64_t>(1) << 16;                     // LBO (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;             // SBO: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                     // SWIZZLE_128B
  return d;
}

// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle.  Atoms
// of 64 16-bit MN elements (128 bytes) x 8 K rows (1024 bytes): `lbo` bytes
// between atoms along MN, `sbo` bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);       // start address
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;   // MN atom stride
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;   // K group stride
  d |= static_cast<uint64_t>(1) << 46;                     // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                     // SWIZZLE_128B
  return d;
}

// Instruction descriptor: D fp32, A/B K-major, M = 128, N = n.
//   kind::f16 with bf16 inputs (a/b format 1), kind::f8f6f4 with e4m3 (0).
__device__ __forceinline__ uint32_t umma_idesc(int n, bool bf16) {
  uint32_t d = 0;
  d |= 1u << 4;                                   // D format: f32
  const uint32_t fmt = bf16 ? 1u : 0u;
  d |= fmt << 7;                                  // A format
  d |= fmt << 10;                                 // B format
  d |= static_cast<uint32_t>(n >> 3) << 17;       // N / 8
  d |= static_cast<uint32_t>(128 >> 4) << 24;     // M / 16
  return d;
}

__device__ __forceinline__ void umma_bf16(uint32_t dtmem, uint64_t adesc,
                                          uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_e4m3(uint32_t dtmem, uint64_t adesc,
                                          uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once every tcgen05 op issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 columns of 32-bit values from the warp's lane quarter.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 columns of 32-bit values: thread t of the warp gets lane
// (quarter * 32 + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the special-function unit (PTX ex2.approx.ftz: 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ conversions
__device__ __forceinline__ float bf16_lo(uint32_t v) {
  return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

__device__ __forceinline__ float bfround(float f) {
  return __bfloat162float(__float2bfloat16_rn(f));
}

// Two e4m3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// Saturating round-to-nearest-even e4m3 encode.
__device__ __forceinline__ uint8_t f2e4m3(float f) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3));
}

// Cached-at-L2-only loads for data other CTAs wrote during this kernel.
__device__ __forceinline__ float ld_cg(const float* p) { return __ldcg(p); }

// Row index (in units of head_dim elements) of (layer, page, K/V, kv head,
// slot) in the paged cache [layer][page][2][n_kv_heads][page_size][head_dim].
__host__ __device__ __forceinline__ size_t kv_row(int layer, int num_pages,
                                                  int n_kv_heads, int page_size,
                                                  int page, int kv, int head,
                                                  int slot) {
  return ((((static_cast<size_t>(layer) * num_pages + page) * 2 + kv) *
               n_kv_heads + head) * page_size) + slot;
}

template <typename T>
__device__ __forceinline__ T* resolve(const DPtr& d, const Binding* b) {
  char* base = static_cast<char*>(d.slot >= 0 ? b->p[d.slot] : d.p);
  return reinterpret_cast<T*>(base + d.offset);
}

}  // namespace dl
