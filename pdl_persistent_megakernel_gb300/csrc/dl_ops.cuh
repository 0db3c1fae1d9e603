// dl_ops.cuh -- the decode step's tile engines.  Each engine runs one CTA's
// share of an operation; the standalone kernels and the megakernel both call
// them (the megakernel once per instruction).
//
// CTA shape: 288 threads.  Warp 0 lane 0 streams operands into a ring of
// shared-memory stages (TMA tiled loads for weights/activations, bulk copies
// for KV pages); warps 1-8 compute.  Pipeline hand-off uses mbarriers
// (full: bytes landed, empty: stage consumed).  A consumer group's leader
// waits on each mbarrier and a named barrier fans the result out, so every
// wait is bounded and a timeout cannot strand threads at a barrier.
//
// Work split (Stream-K): an operation's work is a line of equal "units" (one
// 128-byte k-block of a 128-row weight tile; one 64-key block of a request's
// KV stream) cut into G contiguous ranges, one per CTA, so every CTA moves the
// same number of bytes.  A tile (or request/kv-head pair) covered by several
// CTAs is finished by the last one to arrive on its counter, which sums the
// partials in CTA order -- deterministic, independent of arrival order.
#pragma once

#include "dl_device.cuh"

namespace dl {

// ----------------------------------------------------------------- waits
// How an operation learns that its inputs are ready: under the standalone
// kernels it is programmatic dependent launch (griddepcontrol.wait, after
// which dependents may launch); inside the megakernel it is acquire-polling
// of event counters that producer instructions release-add.
struct Dep {
  int mode;  // 0: griddepcontrol, 1: counters
  int n;
  const unsigned* ev[4];
  unsigned val[4];
};

__device__ __forceinline__ bool poll_deps(const Dep& d, const KernelCtx& ctx,
                                          unsigned where) {
  for (int i = 0; i < d.n; ++i)
    if (!wait_counter(d.ev[i], d.val[i], ctx, where)) return false;
  fence_proxy_async_global();
  return true;
}

// One thread's wait before its first dependent access.
__device__ __forceinline__ bool single_wait(const Dep& d, const KernelCtx& ctx,
                                            unsigned where) {
  if (d.mode == 0) {
    gdc_wait();
    gdc_launch_dependents();
    return !aborted(ctx.status);
  }
  return poll_deps(d, ctx, where);
}

// A group of nthr threads (named barrier bar_id): the leader polls, the
// barrier fans out; under PDL every thread passes griddepcontrol itself.
__device__ __forceinline__ bool group_wait(const Dep& d, const KernelCtx& ctx,
                                           int bar_id, int nthr, bool leader,
                                           unsigned where, int* sflag) {
  if (d.mode == 0) {
    gdc_wait();
    gdc_launch_dependents();
    return !aborted(ctx.status);
  }
  if (leader) *sflag = poll_deps(d, ctx, where) ? 1 : 0;
  named_bar(bar_id, nthr);
  return *sflag != 0;
}

// Threads that touch no dependent data still pass griddepcontrol once, so
// the CTA's completion implies its dependencies' completion.
__device__ __forceinline__ void idle_wait(const Dep& d) {
  if (d.mode == 0) {
    gdc_wait();
    gdc_launch_dependents();
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------ Stream-K ranges
// Unit counts stay below 2^32 / G (checked when a plan is made), so the
// range arithmetic is 32-bit: 64-bit division is a long emulated sequence.
__device__ __forceinline__ int sk_begin(int U, int G, int c) {
  return static_cast<int>((static_cast<unsigned>(U) * static_cast<unsigned>(c)) /
                          static_cast<unsigned>(G));
}

// The CTA whose range holds unit x (the last CTA whose range starts <= x).
__device__ __forceinline__ int sk_owner(int U, int G, int x) {
  int c = static_cast<int>((static_cast<unsigned>(x) * static_cast<unsigned>(G)) /
                           static_cast<unsigned>(U));
  if (c >= G) c = G - 1;
  while (c > 0 && sk_begin(U, G, c) > x) --c;
  while (c + 1 < G && sk_begin(U, G, c + 1) <= x) ++c;
  return c;
}

// L2 prefetch of the first `pf.units` units of the next projection's share
// c (its weight tiles; the activations do not exist yet).  One thread.
__device__ __forceinline__ void prefetch_next_share(const PrefetchSpec& pf, int c) {
  if (!pf.tmap || c >= pf.G) return;
  const int U = pf.NT * pf.KB;
  const int u0 = sk_begin(U, pf.G, c), u1 = sk_begin(U, pf.G, c + 1);
  for (int u = u0; u < u1 && u < u0 + pf.units; ++u) {
    const int t = pf.t_base + u / pf.KB, kb = u % pf.KB;
    tma_prefetch_l2_2d(pf.tmap, kb * pf.kel, t * 128);
    if (pf.pair) tma_prefetch_l2_2d(pf.tmap, kb * pf.kel, pf.up_row + t * 128);
  }
}

__device__ __forceinline__ int sk_contributors(int U, int G, int ts, int len, int* ctb);
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi);

// =================================================================== NORM
// Residual add + RMSNorm (+ per-token, per-128-group e4m3 quantisation):
//   r = bf16(x + res);  h = r * rsqrt(mean(r^2) + eps) * w
// One CTA handles rows [c * rows_per_cta, ...); 256 consumer threads, 16-byte
// vectors, H <= 8192.  With the producing projection's Stream-K partials
// (a.part), x is first formed here: the partials of the CTAs whose ranges
// hold each tile, summed in CTA order (the order of the projection's own
// fix-up) and rounded to bf16; x is written out as well.
constexpr int kNormTabOff = 256;                    // contributor table [H/128][1 + kMaxPartContrib]
constexpr int kNormWOff = kNormTabOff + 64 * (1 + kMaxPartContrib) * 4;   // norm weight, bf16 [H]

// x of two of a thread's 8-column vectors (v0, v1; row m), each the bf16 of
// the CTA-ordered sum of its tile's partials: every contributor of both
// vectors, up to six per pass, is loaded before any is added (one round
// trip for the usual five or six contributors of a tile).
__device__ __forceinline__ void norm_partial_sum2(const NormArgs& a, const int* ptab, int m,
                                                  int v0, int v1, bool act0, bool act1,
                                                  uint4& x0, uint4& x1) {
  constexpr int kB = 6;
  const int* tb0 = ptab + (v0 >> 4) * (1 + kMaxPartContrib);
  const int* tb1 = ptab + (v1 >> 4) * (1 + kMaxPartContrib);
  const int n0 = act0 ? tb0[0] : 0, n1 = act1 ? tb1[0] : 0;
  const size_t pstride = static_cast<size_t>(a.part_mp) * 128;
  const size_t r0 = static_cast<size_t>(m) * 128 + ((v0 & 15) << 3);
  const size_t r1 = static_cast<size_t>(m) * 128 + ((v1 & 15) << 3);
  float4 s[2][2];
#pragma unroll
  for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int nn = max(n0, n1);
  for (int k0 = 0; k0 < nn; k0 += kB) {
    float4 l[2][kB][2];
#pragma unroll
    for (int kk = 0; kk < kB; ++kk) {
      if (k0 + kk < n0) {
        const float4* src = reinterpret_cast<const float4*>(
            a.part + static_cast<size_t>(tb0[1 + k0 + kk]) * pstride + r0);
        l[0][kk][0] = __ldcg(src);
        l[0][kk][1] = __ldcg(src + 1);
      }
      if (k0 + kk < n1) {
        const float4* src = reinterpret_cast<const float4*>(
            a.part + static_cast<size_t>(tb1[1 + k0 + kk]) * pstride + r1);
        l[1][kk][0] = __ldcg(src);
        l[1][kk][1] = __ldcg(src + 1);
      }
    }
#pragma unroll
    for (int kk = 0; kk < kB; ++kk) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        if (k0 + kk < (i == 0 ? n0 : n1)) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (k0 + kk == 0) {
              s[i][h] = l[i][kk][h];
            } else {
              s[i][h].x += l[i][kk][h].x;
              s[i][h].y += l[i][kk][h].y;
              s[i][h].z += l[i][kk][h].z;
              s[i][h].w += l[i][kk][h].w;
            }
          }
        }
      }
    }
  }
  x0 = make_uint4(pack_bf16(s[0][0].x, s[0][0].y), pack_bf16(s[0][0].z, s[0][0].w),
                  pack_bf16(s[0][1].x, s[0][1].y), pack_bf16(s[0][1].z, s[0][1].w));
  x1 = make_uint4(pack_bf16(s[1][0].x, s[1][0].y), pack_bf16(s[1][0].z, s[1][0].w),
                  pack_bf16(s[1][1].x, s[1][1].y), pack_bf16(s[1][1].z, s[1][1].w));
}

// The row's sum of squares over a cluster of kS CTAs: thread ct 0 pushes
// this CTA's part `v` into slot [rank] of every cluster CTA (st.async,
// completing as transaction bytes on that CTA's exchange barrier), then
// every thread waits for its own barrier and adds the kS slots in rank
// order.  One round trip, against two cluster barriers and a remote load.
// Every CTA of the cluster calls this once per launch (an aborted one with
// v = 0), and none exits before the peers' pushes into it have landed, so
// the wait ignores the abort flag; it is bounded by the budget all the same.
template <int kS>
__device__ __forceinline__ float cluster_row_sum(float v, float* xsum, uint64_t* xbar, int ct,
                                                 int rank, const KernelCtx& ctx) {
  cluster_wait();   // every exchange barrier of the cluster is initialised
  if (ct == 0) {
    mbar_arrive_expect_tx(xbar, kS * 4);
    const uint32_t slot = smem_u32(xsum + rank), bar = smem_u32(xbar);
#pragma unroll
    for (int r = 0; r < kS; ++r)
      st_async_f32(cluster_map(slot, static_cast<uint32_t>(r)), v,
                   cluster_map(bar, static_cast<uint32_t>(r)));
  }
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait<true>(xbar, 0)) {
    if (globaltimer() - t0 > ctx.budget_ns) {
      if (ct == 0) report_error(ctx.status, DERR_TIMEOUT, ctx.op_id, blockIdx.x, 40, 0);
      break;
    }
  }
  float tot = 0.f;
#pragma unroll
  for (int r = 0; r < kS; ++r) tot += xsum[r];
  return tot;
}

// NV = 16-byte vectors per thread and row part: 1 (up to 2048 columns), 2
// (4096) or 4 (8192); the registers a thread holds scale with it.
// kS > 1: a row is split over a cluster of kS CTAs (CTA c: row c / kS,
// columns of part c % kS = its cluster rank), which add their sums of
// squares through distributed shared memory (cluster_row_sum; one row per
// CTA, the launch shape the host gives a split norm).  The partial sums of a
// deferred fix-up then spread over kS SMs: one SM keeps only so many loads
// in flight, and a whole row's partials (about 100 KB at H = 4096) took it
// several microseconds.
template <int NV, bool kPart = true, int kS = 1>
__device__ void norm_op(const NormArgs& a, int c, const Dep& dep,
                        const KernelCtx& ctx, uint8_t* smem) {
  const int tid = threadIdx.x;
  float* xsum = reinterpret_cast<float*>(smem + 160);      // [kS] the cluster's sums of squares
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + 192);   // their exchange barrier
  if constexpr (kS > 1) {
    // the exchange barrier is initialised before this CTA's threads arrive
    // on the cluster barrier, which every peer waits on before its push
    if (tid == 32) {
      mbar_init(xbar, 1);
      fence_barrier_init();
    }
    cluster_arrive();
  }
  if (tid < 32) {
    if constexpr (kS > 1) cluster_wait();
    idle_wait(dep);
    return;
  }
  const int ct = tid - 32, lane = tid & 31, wc = ct >> 5;
  if (ct == 0) trace_stamp(ctx, c, TR_START);
  const int split = a.split > 1 ? a.split : 1;
  if (kS == 1 && c % split != 0) {
    // megakernel, a split row: the share of part 0 norms it whole
    if (!group_wait(dep, ctx, 1, 256, ct == 0, 1, reinterpret_cast<int*>(smem + 128))) return;
    if (ct == 0) {
      trace_stamp(ctx, c, TR_DEPS);
      trace_put(ctx, c, TR_UNITS, 0ull);
      trace_stamp(ctx, c, TR_END);
    }
    return;
  }
  float* red = reinterpret_cast<float*>(smem);     // [2][8]
  int* sflag = reinterpret_cast<int*>(smem + 128);
  int* ptab = reinterpret_cast<int*>(smem + kNormTabOff);
  const int H = a.H;
  // this CTA's vectors of 8 columns: [vb, vb + nvec)
  const int nvec = (H >> 3) / kS, vb = (kS > 1 ? c % kS : 0) * nvec;
  // the contributor lists are plain range arithmetic: built before the wait
  if (kPart && a.part) {
    for (int t = (vb >> 4) + ct; t < ((vb + nvec) >> 4); t += 256)
      ptab[t * (1 + kMaxPartContrib)] =
          sk_contributors(a.part_U, a.part_G, t * a.part_KB, a.part_KB, ptab + t * (1 + kMaxPartContrib) + 1);
    named_bar(1, 256);
  }
  // the norm weight does not depend on the previous op: staged in shared
  // memory (each thread its own vectors) before the wait
  const uint16_t* w = static_cast<const uint16_t*>(a.w);
  uint4* wsm = reinterpret_cast<uint4*>(smem + kNormWOff);
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (ct + j * 256 < nvec)
      wsm[vb + ct + j * 256] = __ldg(reinterpret_cast<const uint4*>(w + (vb + ct + j * 256) * 8));
  bool live = group_wait(dep, ctx, 1, 256, ct == 0, 1, sflag);
  // under griddepcontrol each thread read the abort flag itself: one
  // verdict for the CTA, so that no thread is left at a barrier
  if (dep.mode == 0) live = !named_bar_or(1, 256, !live);
  if (!live) {
    if constexpr (kS > 1) cluster_row_sum<kS>(0.f, xsum, xbar, ct, c % kS, ctx);
    return;
  }
  if (ct == 0) trace_stamp(ctx, c, TR_DEPS);
  const Binding* bd = ctx.binding;
  const uint16_t* x = resolve<const uint16_t>(a.x, bd);
  const uint16_t* res = resolve<const uint16_t>(a.res, bd);
  uint16_t* rout = resolve<uint16_t>(a.r_out, bd);
  const int m0 = (c / split) * a.rows_per_cta;
  const int m1 = min(a.M, m0 + (kS > 1 ? 1 : a.rows_per_cta));
  const uint64_t pol_keep = policy_evict_last();
  for (int m = m0; m < m1; ++m) {
    // every load of the row goes out before any store (a store to the
    // residual or x buffer could alias a later load): one round trip
    uint4 xv[NV], rv[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vl = ct + j * 256, v = vb + vl;
      rv[j] = make_uint4(0, 0, 0, 0);
      xv[j] = rv[j];
      if (vl < nvec) {
        const size_t off = static_cast<size_t>(m) * H + v * 8;
        rv[j] = __ldcg(reinterpret_cast<const uint4*>(res + off));
        if (!(kPart && a.part)) xv[j] = __ldcg(reinterpret_cast<const uint4*>(x + off));
      }
    }
    if (kPart && a.part) {
#pragma unroll
      for (int j = 0; j < NV; j += 2) {
        const int vl0 = ct + j * 256, v0 = vb + vl0, v1 = v0 + 256;
        uint4 spare;
        if (vl0 < nvec)
          norm_partial_sum2(a, ptab, m, v0, v1, true, j + 1 < NV && vl0 + 256 < nvec, xv[j],
                            j + 1 < NV ? xv[(j + 1) % NV] : spare);
      }
    }
    // r = bf16(x + res), kept as packed bf16 (exact)
    uint32_t rp[NV][4];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vl = ct + j * 256, v = vb + vl;
      if (vl < nvec) {
        const size_t off = static_cast<size_t>(m) * H + v * 8;
        if (kPart && a.part) *reinterpret_cast<uint4*>(const_cast<uint16_t*>(x) + off) = xv[j];
        const uint32_t xs[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        const uint32_t rs[4] = {rv[j].x, rv[j].y, rv[j].z, rv[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = bfround(bf16_lo(xs[e]) + bf16_lo(rs[e]));
          const float a1 = bfround(bf16_hi(xs[e]) + bf16_hi(rs[e]));
          ss += a0 * a0 + a1 * a1;
          rp[j][e] = static_cast<uint32_t>(f2bf(a0)) |
                     (static_cast<uint32_t>(f2bf(a1)) << 16);
        }
        // the new residual is read again by the next norm, after the
        // projections and the attention have streamed their operands
        // (evict-first) through L2: kept there with evict-last priority
        st_global_v4_hint(rout + off, make_uint4(rp[j][0], rp[j][1], rp[j][2], rp[j][3]), pol_keep);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) rp[j][e] = 0u;
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[(m & 1) * 8 + wc] = ss;
    named_bar(1, 256);
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += red[(m & 1) * 8 + i];
    // the row's sum of squares: the cluster's parts, in rank order
    if constexpr (kS > 1) tot = cluster_row_sum<kS>(tot, xsum, xbar, ct, c % kS, ctx);
    const float inv = rsqrtf(tot / static_cast<float>(H) + a.eps);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int vl = ct + j * 256, v = vb + vl;
      const bool act = vl < nvec;
      float h[8];
      if (act) {
        const uint4 wj = wsm[v];
        const uint32_t ws[4] = {wj.x, wj.y, wj.z, wj.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[2 * e] = bf16_lo(rp[j][e]) * inv * bf16_lo(ws[e]);
          h[2 * e + 1] = bf16_hi(rp[j][e]) * inv * bf16_hi(ws[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) h[e] = 0.f;
      }
      const size_t off = static_cast<size_t>(m) * H + v * 8;
      if (!a.fp8) {
        if (act) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = static_cast<uint32_t>(f2bf(h[2 * e])) |
                   (static_cast<uint32_t>(f2bf(h[2 * e + 1])) << 16);
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.h_out) + off) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
        // 16 consecutive lanes hold one 128-element group
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(h[e]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float s = amax > 0.f ? amax / 448.f : 1.f;
        if (act) {
          uint32_t lo = 0, hi = 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) lo |= static_cast<uint32_t>(f2e4m3(h[e] / s)) << (8 * e);
#pragma unroll
          for (int e = 0; e < 4; ++e) hi |= static_cast<uint32_t>(f2e4m3(h[4 + e] / s)) << (8 * e);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.h_out) + off) = make_uint2(lo, hi);
          if ((v & 15) == 0) a.h_scale[static_cast<size_t>(m) * (H >> 7) + (v >> 4)] = s;
        }
      }
    }
  }
  if (ct == 0) {
    trace_put(ctx, c, TR_UNITS, static_cast<unsigned long long>(c % split == 0 && m1 > m0 ? m1 - m0 : 0));
    trace_stamp(ctx, c, TR_END);
  }
}

// =================================================================== GEMM
constexpr int kMaxTmemBufs = 4;   // TMEM accumulator ring depth (tcgen05 path)

struct GemmSmem {
  int w_bytes, x_bytes, stage_bytes, tile_off, sx_off, sw_off, epi_off, bar_off,
      misc_off, total;
};

constexpr int kMaxContrib = 256;  // CTAs that may share one tile / KV pair

// Finished-tile buffers of the tcgen05 path: two (the epilogue warps fill
// one while the fix-up warps finish the other) when a tile takes at most 16
// KiB, else one.
__host__ __device__ inline int gemm_ntout(int npair, int Mp) {
  return npair * Mp * 128 * 4 <= 16384 ? 2 : 1;
}

// Shared-memory layout of one GEMM CTA: the operand ring, the finished tile,
// the FP8 scales of the current tile run (staged once per run), the QKV
// epilogue's per-token positions / cache rows / RoPE rows, barriers and a
// small control area (flags, contributor list of a Stream-K fix-up).
__host__ __device__ inline GemmSmem gemm_smem_layout(int npair, int Mp, int stages,
                                                     int KB, int fp8, int epi, int M,
                                                     int share) {
  GemmSmem L;
  L.w_bytes = 16384;
  L.x_bytes = ((Mp * 128 + 1023) / 1024) * 1024;
  // 32 KiB of tiles (gate + up, or two consecutive units), then one
  // activation slice per unit
  L.stage_bytes = 2 * L.w_bytes + (npair == 1 ? 2 : 1) * L.x_bytes;
  L.tile_off = stages * L.stage_bytes;
  L.sx_off = L.tile_off + gemm_ntout(npair, Mp) * npair * Mp * 128 * 4;
  L.sw_off = L.sx_off + (fp8 ? KB * Mp * 4 : 0);
  L.epi_off = ((L.sw_off + (fp8 ? 2 * share * 4 : 0)) + 15) & ~15;   // sw [2][share]
  L.bar_off = L.epi_off + (epi == EPI_QKV_ROPE ? M * (8 + 512) + 256 * 4 + 16 : 0);
  L.bar_off = (L.bar_off + 15) & ~15;
  L.misc_off = L.bar_off + (2 * kMaxStages + 2 * kMaxTmemBufs + 5) * 8;
  // two control areas (flags + contributor list): the fix-up warps' and the
  // epilogue warps' (which finish the last tile themselves)
  L.total = L.misc_off + 2 * (256 + kMaxContrib * 4);
  return L;
}

struct GemmShared {
  uint8_t* stage0;
  float* tout;
  float* sx;      // [run][M] activation scales of the current tile run
  float* sw;      // [2][run] weight scales of the current tile run
  int* tok_pos;   // [M] positions (QKV epilogue)
  int* tok_row;   // [M] cache row of (layer, page, K, head 0, slot) (QKV epilogue)
  float2* rope;   // [M][64] (cos, sin) at each token's position (QKV epilogue)
  float* qkw;     // [2][128] q and k head-norm weights (QKV epilogue)
  uint16_t** kvp; // the paged cache, resolved from the binding (QKV epilogue)
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* tready;  // [2] finished tile buffer b written (4 epilogue warps)
  uint64_t* tfree;   // [2] tile buffer b finished and free (2 fix-up warps)
  uint64_t* tprep;   // QKV epilogue operands staged (fix-up warps), or NULL

  int* flag;      // [4]
  int* ctb;       // [kMaxContrib] contributor list of a fix-up
  int* flag2;     // the epilogue warps' own control area (last tile)
  int* ctb2;
};

// dst (the first partial) plus `nc` fp32 partials (float4 granular, nel4
// float4s each) listed in ctb as workspace slot indices, in list order, into
// dst.  Each thread owns up to 8 float4s per pass and loads them for two
// contributors at a time, so a pass costs about nc / 2 L2 round trips.  When
// a thread owns at most 4 float4s and there are more than two partials, it
// loads four contributors at a time instead (one round trip up to four).
template <bool kWide>
__device__ __forceinline__ void ordered_sum4(float4* dst, const float* ws, size_t part,
                                             const int* ctb, int nc, int nel4, int nthr,
                                             int ct) {
  if (kWide && nc > 2 && nel4 <= 4 * nthr) {
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e4 = ct + q * nthr;
      acc[q] = e4 < nel4 ? dst[e4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int j = 0; j < nc; j += 4) {
      float4 v[4][4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float4* src = reinterpret_cast<const float4*>(
            ws + static_cast<size_t>(ctb[j + jj < nc ? j + jj : j]) * part);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e4 = ct + q * nthr;
          v[jj][q] = (j + jj < nc && e4 < nel4) ? __ldcg(src + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (j + jj < nc) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[q].x += v[jj][q].x;
            acc[q].y += v[jj][q].y;
            acc[q].z += v[jj][q].z;
            acc[q].w += v[jj][q].w;
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e4 = ct + q * nthr;
      if (e4 < nel4) dst[e4] = acc[q];
    }
    return;
  }
  constexpr int kQ = 8;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 * nthr < nel4; q0 += kQ) {
    float4 acc[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int e4 = ct + (q0 + q) * nthr;
      acc[q] = e4 < nel4 ? dst[e4] : z;
    }
    for (int j = 0; j < nc; j += 2) {
      const float4* s0 = reinterpret_cast<const float4*>(ws + static_cast<size_t>(ctb[j]) * part);
      const float4* s1 = j + 1 < nc
          ? reinterpret_cast<const float4*>(ws + static_cast<size_t>(ctb[j + 1]) * part) : nullptr;
      float4 v0[kQ], v1[kQ];
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int e4 = ct + (q0 + q) * nthr;
        v0[q] = e4 < nel4 ? __ldcg(s0 + e4) : z;
        v1[q] = (s1 && e4 < nel4) ? __ldcg(s1 + e4) : z;
      }
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        acc[q].x += v0[q].x;
        acc[q].y += v0[q].y;
        acc[q].z += v0[q].z;
        acc[q].w += v0[q].w;
        if (s1) {
          acc[q].x += v1[q].x;
          acc[q].y += v1[q].y;
          acc[q].z += v1[q].z;
          acc[q].w += v1[q].w;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int e4 = ct + (q0 + q) * nthr;
      if (e4 < nel4) dst[e4] = acc[q];
    }
  }
}

// Stream-K bookkeeping shared by the GEMM fix-up and the attention combine:
// write the list of CTAs whose ranges intersect units [ts, ts + len) (in
// CTA order, as workspace slot indices c * 2 + slot) and return its size.
__device__ __forceinline__ int sk_contributors(int U, int G, int ts, int len,
                                               int* ctb) {
  const int cf = sk_owner(U, G, ts), cl = sk_owner(U, G, ts + len - 1);
  int n = 0;
  for (int cc = cf; cc <= cl && n < kMaxContrib; ++cc) {
    const int b0 = sk_begin(U, G, cc);
    if (sk_begin(U, G, cc + 1) <= b0) continue;
    ctb[n++] = cc * 2 + ((b0 >= ts) ? 0 : 1);
  }
  return n;
}

// ------------------------------------------------------- GEMM epilogues
// tout = the finished tile: [npair][Mp][128] fp32 (rows of the weight tile on
// the fast axis).  nthr threads (128 or 256) with group barrier `bar`; the
// per-token epilogues run one warp per token, lane l holding elements
// l, l + 32, l + 64, l + 96.

__device__ void epi_store_bf16(const GemmArgs& a, int tg, const float* tout,
                               int nthr, int ct, const Binding* bd) {
  uint16_t* out = resolve<uint16_t>(a.out, bd);
  for (int e = ct; e < a.M * 32; e += nthr) {
    const int m = e >> 5, i = (e & 31) * 4;
    const float4 v = *reinterpret_cast<const float4*>(tout + m * 128 + i);
    const uint32_t lo = static_cast<uint32_t>(f2bf(v.x)) | (static_cast<uint32_t>(f2bf(v.y)) << 16);
    const uint32_t hi = static_cast<uint32_t>(f2bf(v.z)) | (static_cast<uint32_t>(f2bf(v.w)) << 16);
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(m) * a.ldo + tg * 128 + i) = make_uint2(lo, hi);
  }
}

// Operands of the QKV epilogue, loaded once per CTA before the dependency
// wait (none is an earlier operation's output): positions, the cache row of
// each token's slot, the (cos, sin) rows at each position, the q / k
// head-norm weights and the cache pointer.  Under load one dependent global
// read costs about a microsecond, so the epilogue itself reads shared memory
// only.  Out-of-range positions or pages are reported and skipped.
__device__ void qkv_epi_prepare(const GemmArgs& a, int nthr, int ct, int bar,
                                const KernelCtx& ctx, const GemmShared& sh) {
  const Binding* bd = ctx.binding;
  const int* pos = resolve<const int>(a.pos, bd);
  const int* bt = resolve<const int>(a.bt, bd);
  for (int m = ct; m < a.M; m += nthr) {
    int p = pos[m];
    int row = -1;
    if (p < 0 || p >= a.rope_max_pos) {
      report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 20, p);
      p = 0;
    } else {
      const int lp = p / a.P;
      const int page = lp < a.max_pages ? bt[static_cast<size_t>(m / a.T) * a.max_pages + lp] : -1;
      if (page < 0 || page >= a.num_pages)
        report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 21, lp);
      else
        row = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, 0, p % a.P));
    }
    sh.tok_pos[m] = p;
    sh.tok_row[m] = row;
  }
  for (int e = ct; e < 256; e += nthr) {
    const uint16_t* w = static_cast<const uint16_t*>(e < 128 ? a.q_norm_w : a.k_norm_w);
    sh.qkw[e] = __uint_as_float(static_cast<uint32_t>(w[e & 127]) << 16);
  }
  if (ct == 0) *sh.kvp = resolve<uint16_t>(a.kv, bd);
  named_bar(bar, nthr);
  const float2* cs = reinterpret_cast<const float2*>(a.rope_cs);
  for (int e = ct; e < a.M * 64; e += nthr)
    sh.rope[e] = cs[static_cast<size_t>(sh.tok_pos[e >> 6]) * 64 + (e & 63)];
  named_bar(bar, nthr);
}

// QK-norm + RoPE (neox pairs i, i + 64) for q and k heads; q heads go to the
// q buffer, k and v heads to their slot in the paged cache.
__device__ void epi_qkv_rope(const GemmArgs& a, int tg, const float* tout,
                             int nthr, int ct, const KernelCtx& ctx,
                             const GemmShared& sh) {
  const int lane = ct & 31, wi = ct >> 5, nw = nthr >> 5;
  uint16_t* kv = *sh.kvp;
  const int hh = tg;
  const bool is_q = hh < a.Hq;
  const bool is_k = !is_q && hh < a.Hq + a.Hkv;
  float wn[4] = {1.f, 1.f, 1.f, 1.f};
  if (is_q || is_k) {
#pragma unroll
    for (int k = 0; k < 4; ++k) wn[k] = sh.qkw[(is_q ? 0 : 128) + lane + 32 * k];
  }
  for (int m = wi; m < a.M; m += nw) {
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = bfround(tout[m * 128 + lane + 32 * k]);
    float o[4];
    if (is_q || is_k) {
      const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
      const float inv = rsqrtf(ss * (1.f / 128.f) + a.eps);
      float xn[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) xn[k] = bfround(v[k] * inv * wn[k]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 cs = sh.rope[m * 64 + lane + 32 * (k & 1)];
        const float partner = xn[k ^ 2];
        o[k] = k < 2 ? xn[k] * cs.x - partner * cs.y : xn[k] * cs.x + partner * cs.y;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = v[k];
    }
    if (is_q) {
      uint16_t* dst = static_cast<uint16_t*>(a.q_out) + (static_cast<size_t>(m) * a.Hq + hh) * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[lane + 32 * k] = f2bf(o[k]);
    } else {
      const int row = sh.tok_row[m];
      if (row < 0) continue;
      const int kvsel = is_k ? 0 : 1;
      const int kh = is_k ? hh - a.Hq : hh - a.Hq - a.Hkv;
      // row addresses (layer, page, K, head 0, slot): V is Hkv * P rows on,
      // head kh is kh * P rows on
      const size_t r = static_cast<size_t>(row) +
                       (static_cast<size_t>(kvsel) * a.Hkv + kh) * a.P;
#pragma unroll
      for (int k = 0; k < 4; ++k) kv[r * 128 + lane + 32 * k] = f2bf(o[k]);
    }
  }
}

__device__ void epi_silu_mul(const GemmArgs& a, int tg, const float* tout,
                             int nthr, int ct) {
  const int lane = ct & 31, wi = ct >> 5, nw = nthr >> 5;
  for (int m = wi; m < a.M; m += nw) {
    float av[4];
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float gv = bfround(tout[m * 128 + lane + 32 * k]);
      const float uv = bfround(tout[(a.Mp + m) * 128 + lane + 32 * k]);
      av[k] = gv / (1.f + expf(-gv)) * uv;
      amax = fmaxf(amax, fabsf(av[k]));
    }
    const size_t base = static_cast<size_t>(m) * a.act_ld + tg * 128;
    if (!a.fp8) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        static_cast<uint16_t*>(a.act)[base + lane + 32 * k] = f2bf(av[k]);
    } else {
      amax = warp_max(amax);
      const float sc = amax > 0.f ? amax / 448.f : 1.f;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        static_cast<uint8_t*>(a.act)[base + lane + 32 * k] = f2e4m3(av[k] / sc);
      if (lane == 0) a.act_scale[static_cast<size_t>(m) * (a.act_ld >> 7) + tg] = sc;
    }
  }
}

// fp32 logits, then per-token (max, lowest index) of this 128-entry tile; the
// last tile to finish reduces all tiles into the greedy ids.
__device__ void epi_logits(const GemmArgs& a, int tg, int tl, const float* tout,
                           int nthr, int ct, int bar, const KernelCtx& ctx,
                           const GemmShared& sh) {
  const Binding* bd = ctx.binding;
  float* logits = resolve<float>(a.out, bd);
  const int lane = ct & 31, wi = ct >> 5, nw = nthr >> 5;
  for (int m = wi; m < a.M; m += nw) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = lane + 32 * k;
      const float v = tout[m * 128 + i];
      logits[static_cast<size_t>(m) * a.ldo + tg * 128 + i] = v;
      if (v > bv || (v == bv && tg * 128 + i < bi)) {
        bv = v;
        bi = tg * 128 + i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      a.best_val[static_cast<size_t>(tl) * a.M + m] = bv;
      a.best_idx[static_cast<size_t>(tl) * a.M + m] = bi;
    }
  }
  __threadfence();
  named_bar(bar, nthr);
  if (ct == 0) {
    const unsigned old = atomicAdd(a.done_cnt, 1u);
    sh.flag[1] = (old + 1 == static_cast<unsigned>(a.NT)) ? 1 : 0;
  }
  named_bar(bar, nthr);
  if (!sh.flag[1]) return;
  __threadfence();
  int* ids = resolve<int>(a.ids, bd);
  for (int m = wi; m < a.M; m += nw) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int t = lane; t < a.NT; t += 32) {
      const float v = __ldcg(a.best_val + static_cast<size_t>(t) * a.M + m);
      const int ix = __ldcg(a.best_idx + static_cast<size_t>(t) * a.M + m);
      if (v > bv || (v == bv && ix < bi)) {
        bv = v;
        bi = ix;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) ids[m] = bi;
  }
  if (ct == 0) *a.done_cnt = 0u;
}

// Finish tile tl (local index; global tg = t_base + tl): Stream-K fix-up,
// then the epilogue.  tout holds this CTA's sum over its k-blocks.
// kWide: the four-contributor sum (the megakernel keeps the two-wide one,
// whose registers its engine functions can spare)
template <bool kWide>
__device__ void gemm_finish_tile(const GemmArgs& a, int c, int u0, int tl,
                                 bool full_tile, int npair, int nthr, int ct,
                                 int bar, const KernelCtx& ctx,
                                 const GemmShared& sh) {
  float* tout = sh.tout;
  const int nel = npair * a.Mp * 128;
  if (a.epi == EPI_PARTIALS) {
    // no fix-up here: the partial goes to slot 0 when this CTA's range
    // begins inside the tile, slot 1 when the tile begins inside it (the
    // slot numbering of sk_contributors); the next op sums the slots
    const int slot = u0 >= tl * a.KB ? 0 : 1;
    float4* mine = reinterpret_cast<float4*>(a.ws + static_cast<size_t>(c * 2 + slot) * nel);
    for (int e4 = ct; e4 < a.M * 32 * npair; e4 += nthr) {
      const int pp = e4 / (a.M * 32), r4 = e4 - pp * a.M * 32;
      mine[pp * a.Mp * 32 + r4] = reinterpret_cast<const float4*>(tout)[pp * a.Mp * 32 + r4];
    }
    named_bar(bar, nthr);  // tout is reused by the next tile
    return;
  }
  if (!full_tile) {
    const int U = a.NT * a.KB;
    const int ts = tl * a.KB;
    // The CTA whose range holds the tile's first unit reaches its part of
    // the tile last (that part ends its range): it finishes the tile.  The
    // others publish their partial early and add an arrival.
    if (u0 > ts) {
      float4* mine = reinterpret_cast<float4*>(a.ws + static_cast<size_t>(c * 2) * nel);
      for (int e4 = ct; e4 < nel / 4; e4 += nthr) mine[e4] = reinterpret_cast<const float4*>(tout)[e4];
      __threadfence();
      named_bar(bar, nthr);
      if (ct == 0) atomicAdd(a.tile_cnt + tl, 1u);
      named_bar(bar, nthr);  // tout is reused by the next tile
      return;
    }
    if (ct == 0) {
      const int n = sk_contributors(U, a.G, ts, a.KB, sh.ctb);
      sh.flag[3] = n;
      const bool ok = n <= 1 || wait_counter(a.tile_cnt + tl, static_cast<unsigned>(n - 1), ctx, 23);
      sh.flag[0] = ok ? 1 : 0;
      a.tile_cnt[tl] = 0u;
    }
    named_bar(bar, nthr);
    if (!sh.flag[0]) return;
    __threadfence();
    // this CTA's partial (first in CTA order) plus the others' in CTA order:
    // the sum does not depend on which CTA finished when
    ordered_sum4<kWide>(reinterpret_cast<float4*>(tout), a.ws, static_cast<size_t>(nel), sh.ctb + 1,
                 sh.flag[3] - 1, nel / 4, nthr, ct);
    if (ct == 0) trace_stamp(ctx, c, TR_REDUCE);
    named_bar(bar, nthr);
  }
  const int tg = a.t_base + tl;
  switch (a.epi) {
    case EPI_QKV_ROPE:
      epi_qkv_rope(a, tg, tout, nthr, ct, ctx, sh);
      break;
    case EPI_STORE_BF16:
      epi_store_bf16(a, tg, tout, nthr, ct, ctx.binding);
      break;
    case EPI_SILU_MUL:
      epi_silu_mul(a, tg, tout, nthr, ct);
      break;
    case EPI_LOGITS:
      epi_logits(a, tg, tl, tout, nthr, ct, bar, ctx, sh);
      break;
    default:
      break;
  }
  named_bar(bar, nthr);  // tout is reused by the next tile
}

// ------------------------------------------------------ GEMV dot products
__device__ __forceinline__ float dot8_bf16(const uint4& w, const uint4& x) {
  float s = 0.f;
  s = fmaf(bf16_lo(w.x), bf16_lo(x.x), s);
  s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
  s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
  s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
  s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
  s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
  s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
  s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
  return s;
}

__device__ __forceinline__ void unpack_e4m3x16(const uint4& v, float* f) {
  const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 lo = e4m3x2_to_f2(static_cast<uint16_t>(ws[e] & 0xFFFF));
    const float2 hi = e4m3x2_to_f2(static_cast<uint16_t>(ws[e] >> 16));
    f[4 * e] = lo.x;
    f[4 * e + 1] = lo.y;
    f[4 * e + 2] = hi.x;
    f[4 * e + 3] = hi.y;
  }
}

// The activation scales [M][KB] of the whole projection input, staged once
// per CTA (float4 loads, several in flight per thread).
// Activation scales [M][KB] -> shared [KB][Mp] (zero for padding tokens):
// an epilogue reads the Mp scales of one k-block as contiguous vectors.
__device__ __forceinline__ void stage_x_scales(const GemmArgs& a, const GemmShared& sh,
                                               int nthr, int ct, int bar, int u0, int nunits) {
  const int M = a.M, KB = a.KB, Mp = a.Mp;
  if (nunits >= KB) {
    for (int e = ct; e < M * KB; e += nthr) {
      const int m = e / KB, kb = e - m * KB;
      sh.sx[kb * Mp + m] = __ldcg(a.x_scale + e);
    }
    for (int e = ct; e < (Mp - M) * KB; e += nthr) {
      const int m = M + e / KB, kb = e % KB;
      sh.sx[kb * Mp + m] = 0.f;
    }
  } else {
    // only the k-blocks of this share's units (a share shorter than a tile
    // touches at most nunits of them), every load of a pass before its
    // stores: the staging sits between the dependency release and the
    // first unit's promotion (down projection: 96 k-blocks, about 20 used)
    for (int e0 = ct; e0 < nunits * Mp; e0 += 4 * nthr) {
      float v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + q * nthr;
        const int i = e / Mp, m = e - i * Mp;
        v[q] = (e < nunits * Mp && m < M) ? __ldcg(a.x_scale + m * KB + (u0 + i) % KB) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + q * nthr;
        const int i = e / Mp, m = e - i * Mp;
        if (e < nunits * Mp) sh.sx[((u0 + i) % KB) * Mp + m] = v[q];
      }
    }
  }
  named_bar(bar, nthr);
}

// Weight scales of every unit of the share [npair][n] (weights are not an
// operation's output: staged before the dependency wait; read after the
// epilogue group's next barrier).
__device__ __forceinline__ void stage_w_scales(const GemmArgs& a, const GemmShared& sh, int u0,
                                               int n, int nthr, int ct) {
  const int npair = a.pair ? 2 : 1;
  for (int e = ct; e < npair * n; e += nthr) {
    const int p = e / n, i = e - p * n;
    const int u = u0 + i;
    const int tg = a.t_base + u / a.KB, kb = u % a.KB;
    const int rt = p == 0 ? tg : (a.up_row >> 7) + tg;
    sh.sw[p * n + i] = __ldg(a.w_scale + static_cast<size_t>(rt) * a.KB + kb);
  }
}

// ------------------------------------------------------------ pipelines
// Where the operands of a pipeline's units live and how they are handed
// over.  Every slot holds 32 KiB of weight tiles or K/V, then activation
// slices: a GEMM slot holds the gate and up tiles of one unit, or, without
// gate/up pairing, the tiles of two consecutive units (ups = 2), each with
// its activation slice; an attention slot holds one 64-key block (K, then
// V).  Streaming two adjacent 128-byte k-blocks of the same weight rows at
// once runs near the HBM copy rate, one at a time about a quarter slower.
// A standalone kernel owns a ring of `ns` slots; the streaming megakernel
// has one ring for all instructions of a worker, filled in queue order by
// its producer warp, and seq0 is the ring sequence number of the share's
// first slot.
// q / d for q < 2^28 and 2 <= d <= 16: the high word of q * ceil(2^32 / d)
// (the error q * (ceil(2^32 / d) - 2^32 / d) / 2^32 stays below 1 / d), so
// the rings never divide by a runtime value.
__host__ __device__ constexpr uint32_t fdiv_magic(uint32_t d) { return 0xFFFFFFFFu / d + 1u; }
__device__ __forceinline__ uint32_t fdiv(uint32_t q, uint32_t magic) { return __umulhi(q, magic); }

struct Pipe {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  uint32_t slot_bytes;
  uint32_t ns;      // slots, >= 2
  uint32_t ns_magic;
  uint32_t seq0;
  int ups;          // units per slot: 1 or 2
  int x_bytes;      // bytes of one unit's activation slice (after the tiles)
  int empty_cnt;    // arrivals that free a slot (1: one MMA commit; 8: 8 warps)
};

constexpr int kSlotTiles = 32768;   // bytes of weight tiles / K+V per slot

__device__ __forceinline__ void pipe_set_ns(Pipe& P, uint32_t ns) {
  P.ns = ns;
  P.ns_magic = fdiv_magic(ns);
}
__device__ __forceinline__ int pipe_sub(const Pipe& P, int i) { return i & (P.ups - 1); }
__device__ __forceinline__ uint32_t pipe_q(const Pipe& P, int i) {
  return P.seq0 + static_cast<uint32_t>(i >> (P.ups - 1));
}
__device__ __forceinline__ uint32_t pipe_idx(const Pipe& P, uint32_t q) {
  return q - fdiv(q, P.ns_magic) * P.ns;
}
__device__ __forceinline__ uint8_t* pipe_slot(const Pipe& P, uint32_t q) {
  return P.base + pipe_idx(P, q) * P.slot_bytes;
}
__device__ __forceinline__ uint64_t* pipe_full(const Pipe& P, uint32_t q) { return P.full + pipe_idx(P, q); }
__device__ __forceinline__ uint64_t* pipe_empty(const Pipe& P, uint32_t q) { return P.empty + pipe_idx(P, q); }
__device__ __forceinline__ uint32_t pipe_par(const Pipe& P, uint32_t q) { return fdiv(q, P.ns_magic) & 1u; }
// unit i of n is the last one of its slot: the slot is released after it
__device__ __forceinline__ bool pipe_last(const Pipe& P, int i, int n) {
  return pipe_sub(P, i) == P.ups - 1 || i == n - 1;
}

// GEMM unit i: weight tile p (gate / up, or the single tile) and the
// activation slice.
__device__ __forceinline__ uint8_t* gemm_w(const Pipe& P, int i, int p) {
  return pipe_slot(P, pipe_q(P, i)) + (pipe_sub(P, i) + p) * 16384;
}
__device__ __forceinline__ uint8_t* gemm_x(const Pipe& P, int i) {
  return pipe_slot(P, pipe_q(P, i)) + kSlotTiles + pipe_sub(P, i) * P.x_bytes;
}

// A warp waits until unit i's slot is full (all lanes poll, the warp agrees);
// false if the wait gave up.
__device__ __forceinline__ bool pipe_warp_wait(const Pipe& P, int i, const KernelCtx& ctx,
                                               unsigned where) {
  const uint32_t q = pipe_q(P, i);
  return warp_wait(pipe_full(P, q), pipe_par(P, q), ctx, where);
}

// TMEM accumulator ring of the tcgen05 path: buffer b of nbuf at column
// base + b * stride; seq0 counts the accumulations before this share.
struct TmemRing {
  uint32_t base;
  int nbuf;         // >= 2
  uint32_t nbuf_magic;
  int stride;
  uint32_t seq0;
  uint32_t rseq0;   // tile runs handed to the fix-up warps before this share
};

// ------------------------------------------------------------ GEMM engine
// kMG: GEMV token bound (1/2/4, CUDA cores); kMp: tcgen05 N (16/32/64).
// Exactly one of them is non-zero.
//
// Roles.  The producer (warp 0 lane 0 of a standalone kernel, or the
// megakernel's producer warp) streams the weight tile(s) and the activation
// slice of each unit into the pipeline (TMA, 128-byte swizzle); before its
// first dependent read it issues the weights of the first units (they do not
// depend on the previous operation).
//   GEMV (M <= 4): warps 1-8 each take 16 rows of a unit, 8 lanes per row.
//   tcgen05 (M > 4): warp 1 lane 0 issues 4 MMAs (K = 32 bytes each) per
//   weight tile into a ring of TMEM accumulators; warps 5-8 read each unit's
//   accumulator (TMEM lane quarter = warp % 4), apply the FP8 block scales
//   and accumulate the tile in registers.
// Waits are per warp (all lanes poll, the warp agrees); a failed wait marks
// the warp dead, it skips work but keeps the barrier sequence, and the group
// agrees on failure with one OR-barrier per tile run.
//
// gemm_consume_t is the consumer side (warps 1-8); gemm_op_t wraps it with
// the standalone kernel's own stages and producer.
template <int kMG, int kMp, bool kWide = true>
__device__ void gemm_consume_t(const GemmArgs& a, int c, const Dep& dep,
                               const KernelCtx& ctx, const GemmShared& sh,
                               const Pipe& P, const TmemRing& TR) {
  constexpr bool kMMA = kMp > 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npair = a.pair ? 2 : 1;
  const int U = a.NT * a.KB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const int nunits = static_cast<int>(u1 - u0);

  if constexpr (!kMMA) {
    // ----------------------------------------------- CUDA-core GEMV (M <= 4)
    const int ct = tid - 32;
    if (ct == 0) {
      trace_stamp(ctx, c, TR_START);
      trace_put(ctx, c, TR_UNITS, static_cast<unsigned long long>(nunits));
    }
    // the QKV epilogue's operands (positions, cache rows, RoPE rows) are
    // step inputs: load them before the dependency wait
    if (a.epi == EPI_QKV_ROPE) qkv_epi_prepare(a, 256, ct, 1, ctx, sh);
    if (a.fp8) stage_w_scales(a, sh, u0, nunits, 256, ct);
    if (!group_wait(dep, ctx, 1, 256, ct == 0, 12, &sh.flag[2])) return;
    if (ct == 0) trace_stamp(ctx, c, TR_DEPS);
    if (a.fp8) stage_x_scales(a, sh, 256, ct, 1, u0, nunits);
    const int c8 = ct & 7, r0 = ct >> 3;
    bool dead = false;
    int i = 0;
    while (i < nunits) {
      const int u = u0 + i;
      const int tl = static_cast<int>(u / a.KB), kb0 = static_cast<int>(u % a.KB);
      const int run = min(nunits - i, a.KB - kb0);
      float acc[2][4][kMG];
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int m = 0; m < kMG; ++m) acc[p][j][m] = 0.f;
      for (int k = 0; k < run; ++k, ++i) {
        if (!dead) dead = !pipe_warp_wait(P, i, ctx, 13);
        if (i == 0 && ct == 0) trace_stamp(ctx, c, TR_FIRST);
        if (dead) continue;
        const uint8_t* xs = gemm_x(P, i);
        uint4 xv[kMG];
#pragma unroll
        for (int m = 0; m < kMG; ++m)
          xv[m] = *reinterpret_cast<const uint4*>(xs + m * 128 + ((c8 ^ (m & 7)) << 4));
        if (!a.fp8) {
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            if (p >= npair) break;
            const uint8_t* wt = gemm_w(P, i, p);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = r0 + 32 * j;
              const uint4 wv = *reinterpret_cast<const uint4*>(wt + r * 128 + ((c8 ^ (r & 7)) << 4));
#pragma unroll
              for (int m = 0; m < kMG; ++m) acc[p][j][m] += dot8_bf16(wv, xv[m]);
            }
          }
        } else {
          // e4m3 x e4m3 in fp32
          float xf[kMG][16];
#pragma unroll
          for (int m = 0; m < kMG; ++m) unpack_e4m3x16(xv[m], xf[m]);
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            if (p >= npair) break;
            const uint8_t* wt = gemm_w(P, i, p);
            const float sw = sh.sw[p * nunits + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = r0 + 32 * j;
              const uint4 wv = *reinterpret_cast<const uint4*>(wt + r * 128 + ((c8 ^ (r & 7)) << 4));
              float wf[16];
              unpack_e4m3x16(wv, wf);
#pragma unroll
              for (int m = 0; m < kMG; ++m) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) d = fmaf(wf[e], xf[m][e], d);
                const float sa = m < a.M ? sh.sx[(kb0 + k) * a.Mp + m] : 0.f;
                acc[p][j][m] = fmaf(d, sw * sa, acc[p][j][m]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0 && pipe_last(P, i, nunits)) mbar_arrive(pipe_empty(P, pipe_q(P, i)));
      }
      // reduce the 8 lanes that share a row, store the tile sum
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        if (p >= npair) break;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int m = 0; m < kMG; ++m) {
            float v = acc[p][j][m];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            if (c8 == 0 && m < a.M) sh.tout[(p * a.Mp + m) * 128 + r0 + 32 * j] = v;
          }
      }
      if (ct == 0 && i == nunits) trace_stamp(ctx, c, TR_LOOP_END);
      if (named_bar_or(1, 256, dead)) return;
      gemm_finish_tile<kWide>(a, c, u0, tl, kb0 == 0 && run == a.KB, npair, 256, ct, 1, ctx, sh);
    }
    if (ct == 0) trace_stamp(ctx, c, TR_END);
  } else {
    // --------------------------------------------- tcgen05 (M > 4, N = kMp)
    // Two issuing threads (warps 1 and 2, lane 0) take alternate slots: one
    // tcgen05.mma costs the issuing thread about 90 ns, and one thread alone
    // would fall behind the weight stream.  Each commits the accumulators of
    // its units and, after a slot's last unit, the slot's release; the
    // epilogue takes the accumulators in unit order.
    if (warp == 1 || warp == 2) {
      // the share's start: stamped before the dependency wait, like the
      // other engines' (the wait returns at the dependency release)
      if (warp == 1 && lane == 0) {
        trace_stamp(ctx, c, TR_START);
        trace_put(ctx, c, TR_UNITS, static_cast<unsigned long long>(nunits));
      }
      idle_wait(dep);
      const int w = warp - 1;
      if (lane == 0) {
        const uint32_t idesc = umma_idesc(kMp, !a.fp8);
        const bool fp8 = a.fp8 != 0;
        const int nslots = (nunits + P.ups - 1) / P.ups;
        uint32_t last_tq = 0;
        bool any_tq = false;
        for (int j = w; j < nslots; j += 2) {
          const uint32_t q = P.seq0 + static_cast<uint32_t>(j);
          // With an odd number of slots a stage's consecutive uses belong to
          // different issuers, and nothing else keeps this issuer from
          // running a whole ring ahead of the other (the TMEM ring only
          // does when it is no deeper than the slot ring): the parity wait
          // on slot q would then match the stage's earlier phase, still
          // the other issuer's slot q - ns.  So first wait until that
          // earlier use has been consumed (its commit frees the stage).
          if (q >= P.ns && !mbar_wait(pipe_empty(P, q - P.ns), pipe_par(P, q - P.ns), ctx, 12)) break;
          if (!mbar_wait(pipe_full(P, q), pipe_par(P, q), ctx, 14)) break;
          const int i0 = j * P.ups, i1 = min(nunits, i0 + P.ups);
          bool ok = true;
          for (int i = i0; i < i1; ++i) {
            const uint32_t tq = TR.seq0 + static_cast<uint32_t>(i);
            const uint32_t tqd = fdiv(tq, TR.nbuf_magic);
            const int b = static_cast<int>(tq - tqd * TR.nbuf);
            if (tq >= static_cast<uint32_t>(TR.nbuf) &&
                !mbar_wait(&sh.tempty[b], (tqd - 1) & 1, ctx, 15)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors built once per operand and advanced by constants
            // (the start-address field counts 16-byte units: +32 bytes of K
            // = +2); a single thread issues every MMA, and per-MMA address
            // arithmetic between them is what bounds its issue rate
            const uint64_t bd0 = umma_desc_sw128(smem_u32(gemm_x(P, i)));
            const uint32_t dbase = TR.base + b * TR.stride;
            for (int p = 0; p < npair; ++p) {
              const uint32_t d = dbase + p * kMp;
              const uint64_t ad0 = umma_desc_sw128(smem_u32(gemm_w(P, i, p)));
              if (fp8) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  umma_e4m3(d, ad0 + 2 * k, bd0 + 2 * k, idesc, k > 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  umma_bf16(d, ad0 + 2 * k, bd0 + 2 * k, idesc, k > 0 ? 1u : 0u);
              }
            }
            umma_commit(&sh.tfull[b]);
            last_tq = tq;
            any_tq = true;
          }
          if (!ok) break;
          uint64_t* e = pipe_empty(P, q);
          umma_commit(e);
          if (P.empty_cnt > 1) mbar_arrive_cnt(e, static_cast<uint32_t>(P.empty_cnt - 1));
        }
        // no MMA may still read shared memory or write TMEM when we leave
        if (any_tq)
          mbar_drain(&sh.tfull[last_tq % TR.nbuf], (last_tq / TR.nbuf) & 1u,
                     ctx.budget_ns);
      }
      return;
    }
    const int ntb = gemm_ntout(npair, kMp);
    const int tile_floats = npair * a.Mp * 128;
    if (warp == 3 || warp == 4) {
      // fix-up warps: the Stream-K fix-up and epilogue of each finished
      // tile, while the epilogue warps already accumulate the next one.
      // They also stage the QKV epilogue's operands (dependent reads of
      // step inputs, several round trips), off the epilogue warps' path to
      // the first unit; the epilogue warps take them before the last tile.
      const int ft = tid - 96;
      if (a.epi == EPI_QKV_ROPE && sh.tprep) {
        qkv_epi_prepare(a, 64, ft, 3, ctx, sh);
        if (ft == 0) mbar_arrive(sh.tprep);
      }
      idle_wait(dep);
      int i = 0;
      uint32_t rq = TR.rseq0;
      while (i < nunits) {
        const int u = u0 + i;
        const int tl = static_cast<int>(u / a.KB), kb0 = static_cast<int>(u % a.KB);
        const int run = min(nunits - i, a.KB - kb0);
        if (i + run == nunits) break;   // the epilogue warps finish the last tile
        const int b = static_cast<int>(rq % ntb);
        if (!warp_wait(&sh.tready[b], (rq / ntb) & 1, ctx, 18)) return;
        if (aborted(ctx.status)) return;
        GemmShared shb = sh;
        shb.tout = sh.tout + b * tile_floats;
        gemm_finish_tile<kWide>(a, c, u0, tl, kb0 == 0 && run == a.KB, npair, 64, ft, 3, ctx, shb);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.tfree[b]);
        i += run;
        ++rq;
      }
      return;
    }
    if (warp < 5) {
      idle_wait(dep);
      return;
    }
    // epilogue warps 5..8: TMEM lane quarter = warp % 4
    const int et = tid - 160;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (a.epi == EPI_QKV_ROPE && !sh.tprep) qkv_epi_prepare(a, 128, et, 2, ctx, sh);
    if (a.fp8) stage_w_scales(a, sh, u0, nunits, 128, et);
    if (!group_wait(dep, ctx, 2, 128, et == 0, 16, &sh.flag[2])) return;
    if (et == 0) trace_stamp(ctx, c, TR_DEPS);
    if (a.fp8) stage_x_scales(a, sh, 128, et, 2, u0, nunits);
    // loop invariants in registers (the arguments may sit in memory that
    // every asm memory clobber below would make the compiler read again)
    const bool fp8 = a.fp8 != 0;
    const uint32_t tl_base = TR.base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t tstride = static_cast<uint32_t>(TR.stride);
    bool dead = false;
    int i = 0;
    uint32_t rq = TR.rseq0;
    while (i < nunits) {
      const int u = u0 + i;
      const int tl = static_cast<int>(u / a.KB), kb0 = static_cast<int>(u % a.KB);
      const int run = min(nunits - i, a.KB - kb0);
      float acc[2][kMp];
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int m = 0; m < kMp; ++m) acc[p][m] = 0.f;
      for (int k = 0; k < run; ++k, ++i) {
        const uint32_t tq = TR.seq0 + static_cast<uint32_t>(i);
        const uint32_t tqd = fdiv(tq, TR.nbuf_magic);
        const int b = static_cast<int>(tq - tqd * TR.nbuf);
        if (!dead) dead = !warp_wait(&sh.tfull[b], tqd & 1, ctx, 17);
        if (i == 0 && et == 0) trace_stamp(ctx, c, TR_FIRST);
        if (dead) continue;
        tc_fence_after();
        const uint32_t tb = tl_base + static_cast<uint32_t>(b) * tstride;
        const float sw0 = fp8 ? sh.sw[i] : 1.f;
        const float sw1 = (fp8 && npair == 2) ? sh.sw[nunits + i] : 1.f;
        const float4* sxk = reinterpret_cast<const float4*>(sh.sx + (kb0 + k) * kMp);
#pragma unroll
        for (int c16 = 0; c16 < kMp / 16; ++c16) {
          // both tiles' accumulators of these 16 tokens, one wait
          float v[2][16];
          tmem_ld16(tb + c16 * 16, v[0]);
          if (npair == 2) tmem_ld16(tb + kMp + c16 * 16, v[1]);
          tmem_wait_ld();
          if (fp8) {
            float sa[16];
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
              const float4 t4 = sxk[c16 * 4 + e4];
              sa[e4 * 4] = t4.x;
              sa[e4 * 4 + 1] = t4.y;
              sa[e4 * 4 + 2] = t4.z;
              sa[e4 * 4 + 3] = t4.w;
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[0][c16 * 16 + e] = fmaf(v[0][e], sw0 * sa[e], acc[0][c16 * 16 + e]);
            if (npair == 2) {
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[1][c16 * 16 + e] = fmaf(v[1][e], sw1 * sa[e], acc[1][c16 * 16 + e]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[0][c16 * 16 + e] += v[0][e];
            if (npair == 2) {
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[1][c16 * 16 + e] += v[1][e];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.tempty[b]);
      }
      // hand the tile to the fix-up warps through buffer b
      const int b = static_cast<int>(rq % ntb);
      if (rq >= static_cast<uint32_t>(ntb) && !dead)
        dead = !warp_wait(&sh.tfree[b], ((rq / ntb) - 1) & 1, ctx, 19);
      if (named_bar_or(2, 128, dead)) return;
      float* tout = sh.tout + b * tile_floats;
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        if (p >= npair) break;
#pragma unroll
        for (int m = 0; m < kMp; ++m)
          if (m < a.M) tout[(p * a.Mp + m) * 128 + row] = acc[p][m];
      }
      if (et == 0 && i == nunits) trace_stamp(ctx, c, TR_LOOP_END);
      if (i == nunits) {
        // the last tile: finished here, 128 threads, own control area (the
        // fix-up warps may still be on the previous one)
        if (a.epi == EPI_QKV_ROPE && sh.tprep && !warp_wait(sh.tprep, 0, ctx, 24)) dead = true;
        if (named_bar_or(2, 128, dead)) return;
        GemmShared shl = sh;
        shl.tout = tout;
        shl.flag = sh.flag2;
        shl.ctb = sh.ctb2;
        gemm_finish_tile<kWide>(a, c, u0, tl, kb0 == 0 && run == a.KB, npair, 128, et, 2, ctx, shl);
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tready[b]);
      ++rq;
    }
    if (et == 0) trace_stamp(ctx, c, TR_END);
  }
}

// Shared-memory pointers of a GEMM share: operand stages at smem (standalone,
// `stages` of them) and the private area after them.
__device__ __forceinline__ GemmShared gemm_shared(const GemmArgs& a, uint8_t* smem, int stages) {
  const int npair = a.pair ? 2 : 1;
  const GemmSmem L = gemm_smem_layout(npair, a.Mp, stages, a.KB, a.fp8, a.epi, a.M, a.share_max);
  GemmShared sh;
  sh.stage0 = smem;
  sh.tout = reinterpret_cast<float*>(smem + L.tile_off);
  sh.sx = reinterpret_cast<float*>(smem + L.sx_off);
  sh.sw = reinterpret_cast<float*>(smem + L.sw_off);
  sh.tok_pos = reinterpret_cast<int*>(smem + L.epi_off);
  sh.tok_row = sh.tok_pos + a.M;
  sh.rope = reinterpret_cast<float2*>(smem + L.epi_off + a.M * 8);
  sh.qkw = reinterpret_cast<float*>(smem + L.epi_off + a.M * (8 + 512));
  sh.kvp = reinterpret_cast<uint16_t**>(smem + L.epi_off + a.M * (8 + 512) + 256 * 4);
  sh.full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  sh.empty = sh.full + kMaxStages;
  sh.tfull = sh.empty + kMaxStages;
  sh.tempty = sh.tfull + kMaxTmemBufs;
  sh.tready = sh.tempty + kMaxTmemBufs;
  sh.tfree = sh.tready + 2;
  sh.tprep = sh.tfree + 2;
  sh.flag = reinterpret_cast<int*>(smem + L.misc_off);
  sh.ctb = reinterpret_cast<int*>(smem + L.misc_off + 256);
  sh.flag2 = reinterpret_cast<int*>(smem + L.misc_off + 256 + kMaxContrib * 4);
  sh.ctb2 = sh.flag2 + 64;
  return sh;
}

// Standalone GEMM share: its own stages, barriers and producer (warp 0).
template <int kMG, int kMp>
__device__ void gemm_op_t(const GemmArgs& a, int c, const Dep& dep,
                          const KernelCtx& ctx, uint8_t* smem,
                          uint32_t tmem_base) {
  constexpr bool kMMA = kMp > 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npair = a.pair ? 2 : 1;
  const GemmSmem L = gemm_smem_layout(npair, a.Mp, a.stages, a.KB, a.fp8, a.epi, a.M, a.share_max);
  const GemmShared sh = gemm_shared(a, smem, a.stages);
  const int U = a.NT * a.KB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const int nunits = static_cast<int>(u1 - u0);
  const int S = a.stages;
  const uint32_t smag = fdiv_magic(static_cast<uint32_t>(S));   // S >= 2
  const int kel = a.fp8 ? 128 : 64;  // elements per k-block
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kMMA ? 1 : 8);
    }
    for (int b = 0; b < kMaxTmemBufs; ++b) {
      mbar_init(&sh.tfull[b], 1);
      mbar_init(&sh.tempty[b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.tready[b], 4);
      mbar_init(&sh.tfree[b], 2);
    }
    mbar_init(sh.tprep, 1);
    sh.flag[0] = sh.flag[1] = sh.flag[3] = 0;
    sh.flag[2] = 1;
    fence_barrier_init();
  }
  __syncthreads();

  const int ups = npair == 1 ? 2 : 1;
  const int nslots = (nunits + ups - 1) / ups;
  if (warp == 0) {
    // ------------------------------------------------------- producer
    // Lanes 1-31 leave at once: a warp whose other lanes sit in
    // griddepcontrol.wait does not run lane 0 either (measured: the weight
    // loads then start only when the previous kernel has finished).  The
    // CTA's other threads pass the dependency, so its completion still
    // implies its dependencies' completion.
    if (lane != 0) return;
    prefetch_tmap(a.tmap_w);
    prefetch_tmap(a.tmap_x);
    const uint32_t ub = npair * 16384 + a.Mp * 128;   // bytes of one unit
    const uint64_t pw = policy_evict_first(), px = policy_evict_last();
    // the weight tiles / activation slices of the units of slot j
    auto load_w = [&](int j, int s) {
      uint8_t* st = sh.stage0 + s * L.stage_bytes;
      for (int i = j * ups; i < nunits && i < (j + 1) * ups; ++i) {
        const int u = u0 + i;
        const int t = a.t_base + static_cast<int>(u / a.KB), kb = static_cast<int>(u % a.KB);
        const int sub = i - j * ups;
        tma_load_2d(st + sub * 16384, a.tmap_w, &sh.full[s], kb * kel, t * 128, pw);
        if (a.pair)
          tma_load_2d(st + 16384, a.tmap_w, &sh.full[s], kb * kel, a.up_row + t * 128, pw);
      }
    };
    auto load_x = [&](int j, int s) {
      uint8_t* st = sh.stage0 + s * L.stage_bytes;
      for (int i = j * ups; i < nunits && i < (j + 1) * ups; ++i) {
        const int kb = static_cast<int>((u0 + i) % a.KB);
        tma_load_2d(st + kSlotTiles + (i - j * ups) * L.x_bytes, a.tmap_x, &sh.full[s], kb * kel,
                    0, px);
      }
    };
    auto units_in = [&](int j) { return min(ups, nunits - j * ups); };
    // weights of the first stages do not depend on the previous op: they go
    // out before the dependency wait (the ablation variants wait first)
    bool ok = true;
    if (a.gdc_mode != 0) ok = single_wait(dep, ctx, 10);
    const int pre = ok ? min(S, nslots) : 0;
    for (int j = 0; j < pre; ++j) {
      mbar_arrive_expect_tx(&sh.full[j], ub * units_in(j));
      load_w(j, j);
    }
    if (a.gdc_mode == 0) ok = single_wait(dep, ctx, 10);
    // activations of the prefetched stages (issued even after a failed wait
    // so that every armed stage completes and can be drained)
    for (int j = 0; j < pre; ++j) load_x(j, j);
    int issued = pre;
    if (ok) {
      for (int j = pre; j < nslots; ++j) {
        const uint32_t jd = fdiv(static_cast<uint32_t>(j), smag);
        const int s = j - static_cast<int>(jd) * S;
        if (!mbar_wait(&sh.empty[s], (jd - 1) & 1, ctx, 11)) break;
        mbar_arrive_expect_tx(&sh.full[s], ub * units_in(j));
        load_w(j, s);
        load_x(j, s);
        issued = j + 1;
      }
    }
    // every load of this share is out: warm L2 with the next projection's
    // first tiles for the share with this CTA index
    if (ok)
      for (int c2 = c; c2 < a.pf.G; c2 += static_cast<int>(gridDim.x)) prefetch_next_share(a.pf, c2);
    // no copy may be in flight when the CTA leaves
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / S) * S;  // last slot issued to stage s
      mbar_drain(&sh.full[s], (last / S) & 1, ctx.budget_ns);
    }
    return;
  }
  Pipe P;
  P.base = sh.stage0;
  P.full = sh.full;
  P.empty = sh.empty;
  P.slot_bytes = static_cast<uint32_t>(L.stage_bytes);
  pipe_set_ns(P, static_cast<uint32_t>(S));
  P.seq0 = 0;
  P.ups = ups;
  P.x_bytes = L.x_bytes;
  P.empty_cnt = kMMA ? 1 : 8;
  TmemRing TR;
  TR.base = tmem_base;
  TR.nbuf = kMMA ? a.tmem_bufs : 2;   // unused by the GEMV path
  TR.nbuf_magic = fdiv_magic(static_cast<uint32_t>(TR.nbuf));
  TR.stride = npair * (kMMA ? kMp : 0);
  TR.seq0 = 0;
  TR.rseq0 = 0;
  gemm_consume_t<kMG, kMp>(a, c, dep, ctx, sh, P, TR);
}

// ============================================================== ATTENTION
struct AttnSmem {
  int stage_bytes, stage_off, q_off, p_off, o_off, xs_off, stat_off, bar_off, tbar_off, misc_off,
      total;
};

constexpr int kOP = 136;   // fp32 row pitch of the merged O tile (bank spread)

// stage: K (d 0-63 | d 64-127) then V (same), each half 64 keys x 128 bytes,
// 128-byte swizzle (TMA), 32 KiB per 64-key unit.
__host__ __device__ inline AttnSmem attn_smem_layout(int QRp, int stages) {
  AttnSmem L;
  const int nmt = QRp / 16;
  L.stage_bytes = 4 * kAttnKeys * 128;
  L.stage_off = 0;
  L.p_off = L.tbar_off = 0;                         // (tcgen05 layout only)
  L.q_off = stages * L.stage_bytes;                 // bf16 [QRp][128], swizzled
  L.o_off = L.q_off + QRp * 256;                    // fp32 [QRp][kOP]
  // partial-score exchange [2][blocks per iteration][8][nmt*8][32]: two
  // 64-key blocks per iteration below 64 query rows, one at 64
  L.xs_off = L.o_off + QRp * kOP * 4;
  L.stat_off = L.xs_off + 2 * 8 * (nmt < 2 ? 2 : nmt) * 8 * 32 * 4;  // m, l per key group, lse, w, pos
  L.bar_off = L.stat_off + (4 * QRp * 2 + QRp * 3) * 4 + 64;
  L.bar_off = (L.bar_off + 15) & ~15;
  // after the barriers: flags, producer page batch [32 units x 4 pages],
  // token positions [64], contributor list, combine weights [kMaxContrib]
  L.misc_off = L.bar_off + 2 * kMaxStages * 8;
  L.total = L.misc_off + 64 + 32 * 4 * 4 + 64 * 4 + kMaxContrib * 4 + kMaxContrib * 4;
  return L;
}

// Layout of the tcgen05 attention share.  Q and the two P buffers come
// first: an M = 128 operand reads 128 rows of 128 bytes from each start,
// and only the first QRp rows are the operand's (the rest alias what follows
// and feed accumulator rows that are never read).
//   Q  [2 d-halves][QRp][128 B]   P  [2][QRp][128 B]   (128-byte swizzle)
//   stages  [S][K lo | K hi | V lo | V hi]   O  fp32 [QRp][kOP]
//   row lse / positions / max / sum [QRp] each; stage, S/P/PV barriers;
//   control area.
__host__ __device__ inline AttnSmem attn_tc_smem_layout(int QRp, int stages) {
  AttnSmem L;
  L.stage_bytes = 4 * kAttnKeys * 128;
  L.q_off = 0;
  L.p_off = 2 * QRp * 128;
  L.stage_off = (4 * QRp * 128 + 1023) & ~1023;
  L.o_off = L.stage_off + stages * L.stage_bytes;
  L.xs_off = L.o_off;                               // (no score exchange)
  // lse, positions, max, sum [QRp]; the split softmax's four partial sums
  L.stat_off = L.o_off + QRp * kOP * 4;
  L.bar_off = (L.stat_off + 8 * QRp * 4 + 15) & ~15;
  // s_full[2] s_free[2] p_full[2] pv_done[2] s_ready[2] s2_free[2]
  L.tbar_off = L.bar_off + 2 * kMaxStages * 8;
  L.misc_off = L.tbar_off + 12 * 8;
  L.total = L.misc_off + 64 + 32 * 4 * 4 + 64 * 4 + kMaxContrib * 4 + kMaxContrib * 4;
  return L;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return static_cast<uint32_t>(f2bf(lo)) | (static_cast<uint32_t>(f2bf(hi)) << 16);
}

// Split-KV GQA decode attention over 64-key blocks.  The G = Hq / Hkv query
// heads of T tokens (QR = T * G rows; row rr = t * G + g is token r * T + t,
// q head h * G + g, causal limit positions[r * T + t]) share one K/V stream.
// Scores are scaled by log2(e) / sqrt(d) so exponentials are base 2.
//
// Warps 1-8 = 4 key groups (16 keys of each block) x 2 head-dim halves.  The
// two warps of a key group each compute the scores of its 16 keys over their
// own half of d and exchange the fp32 partial sums through shared memory, so
// both hold S = S_lo + S_hi.  Each warp keeps its own online-softmax state
// (row max m, row sum l) in registers, rescales its O slice and adds P V for
// its 64 columns, reusing the S fragments as the A operand.  At the end of a
// (request, kv-head) run the four key groups are merged in a fixed order; a
// run covering only part of the KV stream leaves its normalised partial O_i
// and lse_i, and the last CTA of the pair combines
//   lse = log sum_i e^{lse_i},  O = sum_i e^{lse_i - lse} O_i
// over the partials in CTA order (deterministic).
// Attention block i of a pipeline: K (d 0-63 | d 64-127), then V.
__device__ __forceinline__ uint8_t* attn_k(const Pipe& P, int i) {
  return pipe_slot(P, pipe_q(P, i));
}
__device__ __forceinline__ uint8_t* attn_v(const Pipe& P, int i) {
  return attn_k(P, i) + 2 * kAttnKeys * 128;
}

// One query row of the attention output (warp-wide: lane l holds columns
// 4 l .. 4 l + 3): bf16, or e4m3 codes with the row's scale (the O
// projection's input quantised per token per 128-group).
__device__ __forceinline__ void attn_write_row(const AttnArgs& a, int r, int h, int G, int rr,
                                               float4 v, int lane) {
  const int t = rr / G, g = rr % G;
  const size_t m = static_cast<size_t>(r) * a.T + t;
  const int hq = h * G + g;
  if (!a.fp8) {
    uint16_t* out = static_cast<uint16_t*>(a.out) + (m * a.Hq + hq) * 128 + lane * 4;
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  } else {
    const float am = warp_max(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    const float sc = am > 0.f ? am / 448.f : 1.f;
    const uint32_t code = static_cast<uint32_t>(f2e4m3(v.x / sc)) |
                          (static_cast<uint32_t>(f2e4m3(v.y / sc)) << 8) |
                          (static_cast<uint32_t>(f2e4m3(v.z / sc)) << 16) |
                          (static_cast<uint32_t>(f2e4m3(v.w / sc)) << 24);
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.out) + (m * a.Hq + hq) * 128 + lane * 4) = code;
    if (lane == 0) a.out_scale[m * a.Hq + hq] = sc;
  }
}

// A finished pair run of this CTA: Ob holds its normalised rows, row_lse
// their log-sum-exp (base 2).  The whole pair: write the attention output;
// otherwise publish the partial (slot 0: the pair where this CTA's range
// begins; slot 1: a later pair, the range's last one) and an arrival; the
// pair is combined once the CTA's range is done (attn_combine).
__device__ void attn_pair_out(const AttnArgs& a, int c, int u0, int p, int blk_a, int blk_b,
                              const float* Ob, const float* row_lse, int* pend, int* npend) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int ct = tid - 32, wc = (tid >> 5) - 1;
  const int QRp = a.QRp, G = a.Hq / a.Hkv;
  const int r = p / a.Hkv, h = p % a.Hkv;
  const bool whole = (blk_a == 0 && blk_b == a.NB);
  if (!whole) {
    const int ps = p * a.NB;
    const int slot = (u0 >= ps) ? 0 : 1;
    const size_t part = static_cast<size_t>(QRp) * 129;
    float* mine = a.ws + static_cast<size_t>(c * 2 + slot) * part;
    for (int e4 = ct; e4 < QRp * 32; e4 += 256)
      reinterpret_cast<float4*>(mine)[e4] =
          *reinterpret_cast<const float4*>(Ob + (e4 >> 5) * kOP + (e4 & 31) * 4);
    for (int rr = ct; rr < QRp; rr += 256) mine[QRp * 128 + rr] = row_lse[rr];
    __threadfence();
    named_bar(1, 256);
    if (ct == 0) atomicAdd(a.pair_cnt + p, 1u);
    pend[(*npend)++] = p;
  } else {
    // the whole pair is this CTA's: write the attention output, one warp
    // per query row
    for (int rr = wc; rr < a.QR; rr += 8)
      attn_write_row(a, r, h, G, rr, *reinterpret_cast<const float4*>(Ob + rr * kOP + lane * 4), lane);
  }
}

// Split-KV combine of the pairs this CTA published partials for (warps
// 1-8, named barrier 1).  False after a failed wait.
__device__ bool attn_combine(const AttnArgs& a, int c, const KernelCtx& ctx, const int* pend,
                             int npend, int* flag, int* ctb) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int ct = tid - 32, wc = (tid >> 5) - 1;
  const int QRp = a.QRp, G = a.Hq / a.Hkv;
  const int U = a.R * a.Hkv * a.NB;
  // ---- split-KV combine, shared by all CTAs of a pair: once every partial
  // of the pair is published, contributor j (CTA order) combines query rows
  // [j * per, (j + 1) * per) by their log-sum-exp weights, in CTA order, and
  // writes them (one warp per row).  The pair's counter counts the n
  // publications, then the n finished slices; the last slice resets it.
  for (int k = 0; k < npend; ++k) {
    const int p = pend[k];
    const int ps = p * a.NB;
    const int r = p / a.Hkv, h = p % a.Hkv;
    const size_t part = static_cast<size_t>(QRp) * 129;
    if (ct == 0) {
      const int n = sk_contributors(U, a.G, ps, a.NB, ctb);
      int j = 0;
      while (j < n && (ctb[j] >> 1) != c) ++j;
      flag[1] = n;
      flag[3] = j;
      flag[0] = wait_counter(a.pair_cnt + p, static_cast<unsigned>(n), ctx, 36) ? 1 : -1;
    }
    named_bar(1, 256);
    if (flag[0] < 0) return false;
    __threadfence();
    const int n = flag[1], jme = flag[3];
    const int per = (a.QR + n - 1) / n;
    const int r1 = min(a.QR, (jme + 1) * per);
    for (int rr = jme * per + wc; rr < r1; rr += 8) {
      // lane j holds contributor j's weight (j < 32, then j + 32)
      float l0 = -INFINITY, l1 = -INFINITY;
      if (lane < n) l0 = __ldcg(a.ws + static_cast<size_t>(ctb[lane]) * part + QRp * 128 + rr);
      if (lane + 32 < n) l1 = __ldcg(a.ws + static_cast<size_t>(ctb[lane + 32]) * part + QRp * 128 + rr);
      const float mx = warp_max(fmaxf(l0, l1));
      const float w0 = (mx == -INFINITY || lane >= n) ? 0.f : exp2f(l0 - mx);
      const float w1 = (mx == -INFINITY || lane + 32 >= n) ? 0.f : exp2f(l1 - mx);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float den = 0.f;
      for (int j0 = 0; j0 < n; j0 += 8) {
        float4 v[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj < n ? j0 + jj : 0;
          v[jj] = __ldcg(reinterpret_cast<const float4*>(a.ws + static_cast<size_t>(ctb[j]) * part +
                                                          static_cast<size_t>(rr) * 128) + lane);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          const float wsrc = __shfl_sync(0xffffffffu, j < 32 ? w0 : w1, j & 31);
          if (j < n) {
            den += wsrc;
            acc.x = fmaf(wsrc, v[jj].x, acc.x);
            acc.y = fmaf(wsrc, v[jj].y, acc.y);
            acc.z = fmaf(wsrc, v[jj].z, acc.z);
            acc.w = fmaf(wsrc, v[jj].w, acc.w);
          }
        }
      }
      const float inv = den > 0.f ? 1.f / den : 0.f;
      attn_write_row(a, r, h, G, rr, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv), lane);
    }
    named_bar(1, 256);
    if (ct == 0) {
      const unsigned old = atomicAdd(a.pair_cnt + p, 1u);
      if (old + 1 == 2u * static_cast<unsigned>(n)) a.pair_cnt[p] = 0u;
      trace_stamp(ctx, c, TR_REDUCE);
    }
  }
  return true;
}

// Consumer side of a tcgen05 attention share (warps 1-8; layout
// attn_tc_smem_layout; 512 TMEM columns: O0 [0, 128), O1 [128, 256),
// S0 [256, 320), S1 [320, 384)).  For valid 64-key block g of the share:
//   warp 2 (lane 0) issues S_g = Q K_g^T into S[g & 1] (M = 128 query rows,
//     of which the first QRp are real, N = 64 keys, K = d in 8 steps);
//   warp 3 (lane 0), once P_g is in shared memory, issues O[g & 1] +=
//     P_g V_g (N = d, K = 64 keys in 4 steps, V read MN-major); its commits
//     release K/V's stage and P's buffer;
//   softmax: blocks alternate between two warps per TMEM lane quarter
//     (rows 0-31: warps 4 and 8; rows 32-63: warps 1 and 5), each with its
//     own running maximum and sum per row and its own O.  A warp reads its
//     rows of S_g, masks them, writes P_g (bf16) and, for a partial block,
//     zeroes the V rows past the context (0-probability keys must add
//     exactly 0).  While a block's maximum is within 2^8 of the running one
//     the running maximum stays (P <= 256; exact in the final
//     normalisation, since the warp's O and sum share it); otherwise it
//     moves and the warp rescales its O in TMEM after its previous block's
//     PV.
// At the end of a pair run the first warp of each pair merges the two
// (maximum, sum, O) into Ob with the rows' log-sum-exp (base 2).
__device__ int attn_consume_tc(const AttnArgs& a, int c, const Dep& dep, const KernelCtx& ctx,
                               uint8_t* smem, const AttnSmem& L, const Pipe& P, uint32_t tmem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QRp = a.QRp, G = a.Hq / a.Hkv;
  uint8_t* qs = smem + L.q_off;
  uint8_t* ps = smem + L.p_off;
  float* Ob = reinterpret_cast<float*>(smem + L.o_off);
  float* row_lse = reinterpret_cast<float*>(smem + L.stat_off);
  int* row_pos = reinterpret_cast<int*>(row_lse + QRp);
  float* row_m1 = reinterpret_cast<float*>(row_pos + QRp);    // second warp's max / sum
  float* row_l1 = row_m1 + QRp;
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + L.tbar_off);
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* pv_done = s_full + 6;
  uint64_t* s_ready = s_full + 8;                              // split softmax
  uint64_t* s2_free = s_full + 10;
  float* row_lk = row_l1 + QRp;       // [4][QRp] the exp warps' partial sums
  // staged S of the split softmax, [2][QRp][68] fp32: 64 scores, the
  // exponent offset -max and the block's rescale factor; it shares its
  // memory with Ob, which is written only after a pair run's last block
  int* flag = reinterpret_cast<int*>(smem + L.misc_off);
  int* ctb = flag + 16 + 32 * 4 + 64;
  const int U = a.R * a.Hkv * a.NB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const Binding* bd = ctx.binding;
  const int ct = tid - 32;
  const int nq = QRp > 32 ? 2 : 1;                   // TMEM lane quarters in use
  const int quarter = warp & 3;
  // Up to 32 query rows (TMEM lanes 0-31, which only the warps of SM
  // sub-partition 0 can read) the softmax is split: warp 4 reads S, takes
  // the row maxima and stages S in shared memory; four exp warps, one per
  // sub-partition (8, 5, 6, 7), exponentiate 16 keys each.  With 64 rows
  // two warps per lane quarter alternate blocks.
  const bool split = QRp <= 32 && a.split_sm;
  const int ek = !split ? -1 : warp == 8 ? 0 : warp == 5 ? 1 : warp == 6 ? 2 : warp == 7 ? 3 : -1;
  // softmax role: quarter 0 -> warps 4 (k = 0), 8 (k = 1); quarter 1 -> warps 1, 5
  const bool is_sm = !split && (quarter < nq) && (warp == 4 || warp == 8 || warp == 1 || warp == 5);
  const int kk_sm = (warp >= 5) ? 1 : 0;             // which of the pair
  const int row = quarter * 32 + lane;
  if (ct == 0) {
    trace_stamp(ctx, c, TR_START);
    trace_put(ctx, c, TR_UNITS, static_cast<unsigned long long>(u1 - u0));
  }
  // the positions are step inputs, not the previous kernel's output: staged
  // before the dependency wait, which then leaves one dependent round trip
  // (the queries) before the first QK^T
  int* pos = ctb + kMaxContrib;             // [R T] token positions
  {
    const int* gpos = resolve<const int>(a.pos, bd);
    for (int m = ct; m < a.R * a.T; m += 256) pos[m] = gpos[m];
  }
  named_bar(1, 256);
  if (!group_wait(dep, ctx, 1, 256, ct == 0, 34, &flag[2])) return -1;
  if (ct == 0) trace_stamp(ctx, c, TR_DEPS);
  const uint16_t* qg = static_cast<const uint16_t*>(a.q);
  const uint32_t qs_u32 = smem_u32(qs), ps_u32 = smem_u32(ps);
  const uint32_t idesc_s = umma_idesc(kAttnKeys, true);
  const uint64_t qd0 = umma_desc_sw128(qs_u32), qd1 = qd0 + QRp * 128 / 16;   // Q d-halves
  const uint32_t idesc_o = umma_idesc(128, true) | (1u << 16);   // B (V) MN-major
  const uint32_t t_o = tmem, t_s = tmem + 256;
  const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
  bool dead = false;
  int i = 0;                                // valid blocks before this run (the producer's slots)
  int pend[2], npend = 0;
  int u = u0;
  while (u < u1) {
    const int p = u / a.NB, blk_a = u % a.NB;
    const int run_end = min(u1, (p + 1) * a.NB);
    const int blk_b = run_end - p * a.NB;
    const int r = p / a.Hkv, h = p % a.Hkv;
    const int ctxr = pos[r * a.T + a.T - 1] + 1;
    const int nvb = (ctxr + kAttnKeys - 1) / kAttnKeys;
    const int n = max(0, min(blk_b, nvb) - blk_a);    // valid blocks of this run
    // this pair's query rows: [d-half][row][128 B], 16-byte chunk c8 of a
    // row at (c8 ^ (row & 7)) (128-byte swizzle); rows QR..QRp-1 zero.
    // All of a thread's loads go out before its stores (one round trip).
    {
      uint4 qv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = ct + k * 256, rr = e >> 4, ch = e & 15;
        qv[k] = make_uint4(0, 0, 0, 0);
        if (e < QRp * 16 && rr < a.QR) {
          const int t = rr / G, g = rr % G;
          const size_t src = (static_cast<size_t>(r * a.T + t) * a.Hq + h * G + g) * 128 + ch * 8;
          qv[k] = __ldcg(reinterpret_cast<const uint4*>(qg + src));
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = ct + k * 256, rr = e >> 4, ch = e & 15;
        if (e < QRp * 16) {
          const int hf = ch >> 3, c8 = ch & 7;
          *reinterpret_cast<uint4*>(qs + hf * QRp * 128 + rr * 128 + ((c8 ^ (rr & 7)) << 4)) = qv[k];
        }
      }
    }
    for (int rr = ct; rr < QRp; rr += 256) row_pos[rr] = rr < a.QR ? pos[r * a.T + rr / G] : -1;
    fence_proxy_async_shared();    // Q, written by threads, is read by the tensor core
    named_bar(1, 256);
    if (warp == 2 || (split && warp == 1)) {
      // --------------------------------------------------- QK^T issuer
      // One thread issues a tcgen05.mma every ~70 ns at best, so with the
      // split softmax (warp 1 otherwise idle) two threads issue QK^T, warp 2
      // the run's even blocks and warp 1 the odd ones: a block and the one
      // two later share an S buffer and an issuer.
      const int jstep = split ? 2 : 1;
      const int jfirst = warp == 1 ? 1 : 0;
      if (lane == 0 && !dead && n > jfirst) {
        int last = -1;
        for (int j = jfirst; j < n; j += jstep) {
          const int g = i + j;
          const uint32_t q = pipe_q(P, g);
          if (!mbar_wait(pipe_full(P, q), pipe_par(P, q), ctx, 80) ||
              (g >= 2 && !mbar_wait(&s_free[g & 1], ((g >> 1) - 1) & 1, ctx, 81))) {
            dead = true;
            break;
          }
          if (g == 0) trace_stamp(ctx, c, TR_FIRST);
          tc_fence_after();
          // descriptors advanced by constants (16-byte units): the d half
          // is QRp * 128 (Q) or 64 * 128 (K) bytes on, each K step 32
          const uint64_t kd0 = umma_desc_sw128(smem_u32(attn_k(P, g)));
          const uint32_t ts = t_s + (g & 1) * kAttnKeys;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16(ts, (kk < 4 ? qd0 : qd1) + 2 * (kk & 3),
                      kd0 + (kk >> 2) * (kAttnKeys * 128 / 16) + 2 * (kk & 3), idesc_s,
                      kk > 0 ? 1u : 0u);
          umma_commit(&s_full[g & 1]);
          last = g;
        }
        // nothing the tensor core still runs may outlive the share
        if (dead && last >= 0) mbar_drain(&s_full[last & 1], (last >> 1) & 1, ctx.budget_ns);
      }
      dead = __shfl_sync(0xffffffffu, dead ? 1 : 0, 0) != 0;
    } else if (warp == 3) {
      // ------------------------------------------------------- PV issuer
      if (lane == 0 && !dead && n > 0) {
        int last = -1;
        for (int j = 0; j < n; ++j) {
          const int g = i + j;
          if (!mbar_wait(&p_full[g & 1], (g >> 1) & 1, ctx, 82)) {
            dead = true;
            break;
          }
          tc_fence_after();
          // keys kk*16 .. +15: two 8-key groups (1024 B apart); the d halves
          // (64 elements each) are 8 KiB apart; descriptors advanced by
          // constants (16-byte units)
          const uint64_t pd0 = umma_desc_sw128(ps_u32 + (g & 1) * QRp * 128);
          const uint64_t vd0 = umma_desc_sw128_mn(smem_u32(attn_v(P, g)), kAttnKeys * 128, 1024);
          // split: one O for the run; else O[g & 1] starts at the run's first
          // block of its parity
          const uint32_t to = split ? t_o : t_o + (g & 1) * 128;
          const bool acc0 = split ? j > 0 : j > 1;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(to, pd0 + 2 * kk, vd0 + kk * (2048 / 16), idesc_o,
                      (acc0 || kk > 0) ? 1u : 0u);
          umma_commit(pipe_empty(P, pipe_q(P, g)));
          umma_commit(&pv_done[g & 1]);
          last = g;
        }
        if (dead && last >= 0) mbar_drain(&pv_done[last & 1], (last >> 1) & 1, ctx.budget_ns);
      }
      dead = __shfl_sync(0xffffffffu, dead ? 1 : 0, 0) != 0;
    } else if (split && warp == 4) {
      // ------------------------------------ split softmax: S reader (rows)
      float* Sst = Ob;
      const int lim = row < QRp ? row_pos[row] : -1;    // rows past QRp: all masked
      const int lim0 = row_pos[0];                       // the pair's first query position
      const float scl = a.scale_log2;
      float m_run = -INFINITY;
      for (int j = 0; j < n && !dead; ++j) {
        const int g = i + j;
        const int k0 = (blk_a + j) * kAttnKeys;
        const int nk = min(kAttnKeys, ctxr - k0);
        if (!warp_wait(&s_full[g & 1], (g >> 1) & 1, ctx, 83)) {
          dead = true;
          break;
        }
        tc_fence_after();
        float sv[kAttnKeys];
#pragma unroll
        for (int c4 = 0; c4 < kAttnKeys / 16; ++c4)
          tmem_ld16(t_s + t_lane + (g & 1) * kAttnKeys + c4 * 16, sv + c4 * 16);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[g & 1]);
        // the block's row maximum (four independent chains); masked keys
        // become -inf, so their probabilities are exactly 0
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (nk == kAttnKeys && k0 + kAttnKeys - 1 <= lim0) {
#pragma unroll
          for (int e = 0; e < kAttnKeys; ++e) mq[e & 3] = fmaxf(mq[e & 3], sv[e]);
        } else {
#pragma unroll
          for (int e = 0; e < kAttnKeys; ++e) {
            sv[e] = (e < nk && k0 + e <= lim) ? sv[e] : -INFINITY;
            mq[e & 3] = fmaxf(mq[e & 3], sv[e]);
          }
        }
        float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        mx = row < QRp ? mx * scl : -INFINITY;
        const bool grow = mx > m_run + 8.f;
        float alpha = 1.f;
        if (grow) {
          alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mx);
          m_run = mx;
        }
        // O holds blocks i .. g - 1 of the run: rescale it once PV_{g-1} is
        // done (the exp warps' P_g, and so PV_g, come after this block's
        // staging below)
        if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const int gp = g - 1;
          if (!warp_wait(&pv_done[gp & 1], (gp >> 1) & 1, ctx, 88)) {
            dead = true;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c16 = 0; c16 < 8; ++c16) {
            float ov[16];
            tmem_ld16(t_o + t_lane + c16 * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= alpha;
            tmem_st16(t_o + t_lane + c16 * 16, ov);
          }
          tmem_wait_st();
          tc_fence_before();
        }
        // staging buffer g & 1 was last read for block g - 2
        if (g >= 2 && !warp_wait(&s2_free[g & 1], ((g >> 1) - 1) & 1, ctx, 89)) {
          dead = true;
          break;
        }
        if (row < QRp) {
          float4* st = reinterpret_cast<float4*>(Sst + ((g & 1) * QRp + row) * 68);
#pragma unroll
          for (int e4 = 0; e4 < kAttnKeys / 4; ++e4)
            st[e4] = make_float4(sv[4 * e4], sv[4 * e4 + 1], sv[4 * e4 + 2], sv[4 * e4 + 3]);
          st[kAttnKeys / 4] = make_float4(m_run == -INFINITY ? 0.f : -m_run, alpha, 0.f, 0.f);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_ready[g & 1]);
      }
      // merge: the four partial sums, then O / l and the rows' lse
      named_bar(5, 160);
      float l = 0.f;
      if (row < QRp) {
#pragma unroll
        for (int k = 0; k < 4; ++k) l += row_lk[k * QRp + row];
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      bool ok = n > 0 && !dead;
      if (ok) {
        const int gl = i + n - 1;      // the last PV into O
        ok = warp_wait(&pv_done[gl & 1], (gl >> 1) & 1, ctx, 86);
        if (!ok) dead = true;
      }
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int c16 = 0; c16 < 8; ++c16) {
          float o[16];
          tmem_ld16(t_o + t_lane + c16 * 16, o);
          tmem_wait_ld();
          if (row < QRp) {
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4)
              *reinterpret_cast<float4*>(Ob + row * kOP + c16 * 16 + e4 * 4) =
                  make_float4(o[e4 * 4] * inv, o[e4 * 4 + 1] * inv, o[e4 * 4 + 2] * inv,
                              o[e4 * 4 + 3] * inv);
          }
        }
        tc_fence_before();
      } else if (row < QRp) {
        for (int e4 = 0; e4 < 32; ++e4)
          *reinterpret_cast<float4*>(Ob + row * kOP + e4 * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (row < QRp) row_lse[row] = l > 0.f ? m_run + log2f(l) : -INFINITY;
    } else if (ek >= 0) {
      // ------------------------- split softmax: exp warp ek, keys 16 ek ..
      const float* Sst = Ob;
      const float scl = a.scale_log2;
      const int lrow = lane;                              // query row (< 32)
      float l_k = 0.f;
      for (int j = 0; j < n && !dead; ++j) {
        const int g = i + j;
        const int k0 = (blk_a + j) * kAttnKeys;
        const int nk = min(kAttnKeys, ctxr - k0);
        if (!warp_wait(&s_ready[g & 1], (g >> 1) & 1, ctx, 90)) {
          dead = true;
          break;
        }
        float sv[16];
        float nmb = 0.f, alpha = 1.f;
        if (lrow < QRp) {
          const float4* st = reinterpret_cast<const float4*>(Sst + ((g & 1) * QRp + lrow) * 68);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 v = st[ek * 4 + q4];
            sv[4 * q4] = v.x;
            sv[4 * q4 + 1] = v.y;
            sv[4 * q4 + 2] = v.z;
            sv[4 * q4 + 3] = v.w;
          }
          const float4 ma = st[kAttnKeys / 4];
          nmb = ma.x;
          alpha = ma.y;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s2_free[g & 1]);
        // P buffer g & 1 was last read by PV_{g-2}
        if (g >= 2 && !warp_wait(&pv_done[g & 1], ((g >> 1) - 1) & 1, ctx, 91)) {
          dead = true;
          break;
        }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float p0 = ex2_approx(fmaf(sv[e], scl, nmb));
          const float p1 = ex2_approx(fmaf(sv[e + 1], scl, nmb));
          s4[(e >> 1) & 3] += p0 + p1;
          pk[e >> 1] = pack_bf16(p0, p1);
        }
        l_k = l_k * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
        if (nk < kAttnKeys && ek == 0) {
          // V rows past the context were not loaded (or are stale)
          uint8_t* vst = attn_v(P, g);
          for (int e = lane; e < (kAttnKeys - nk) * 16; e += 32) {
            const int key = nk + (e >> 4), hf = (e >> 3) & 1, c8 = e & 7;
            *reinterpret_cast<uint4*>(vst + hf * kAttnKeys * 128 + key * 128 + c8 * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        if (lrow < QRp) {
          uint8_t* prow = ps + (g & 1) * QRp * 128 + lrow * 128;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int c8 = 2 * ek + h2;
            *reinterpret_cast<uint4*>(prow + ((c8 ^ (lrow & 7)) << 4)) =
                make_uint4(pk[4 * h2], pk[4 * h2 + 1], pk[4 * h2 + 2], pk[4 * h2 + 3]);
          }
        }
        fence_proxy_async_shared();   // P and the zeroed V rows feed the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g & 1]);
      }
      if (lrow < QRp) row_lk[ek * QRp + lrow] = l_k;
      named_bar(5, 160);
    } else if (is_sm) {
      // --------------------------------------------------- softmax warps
      const int lim = row < QRp ? row_pos[row] : -1;    // rows past QRp: all masked
      const int lim0 = row_pos[0];                       // the pair's first query position
      const float scl = a.scale_log2;
      const uint32_t t_my = t_o + static_cast<uint32_t>(((i + kk_sm) & 1) * 128) + t_lane;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = kk_sm; j < n && !dead; j += 2) {
        const int g = i + j;
        const int k0 = (blk_a + j) * kAttnKeys;
        const int nk = min(kAttnKeys, ctxr - k0);
        if (!warp_wait(&s_full[g & 1], (g >> 1) & 1, ctx, 83)) {
          dead = true;
          break;
        }
        tc_fence_after();
        float sv[kAttnKeys];
#pragma unroll
        for (int c4 = 0; c4 < kAttnKeys / 16; ++c4)
          tmem_ld16(t_s + t_lane + (g & 1) * kAttnKeys + c4 * 16, sv + c4 * 16);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[g & 1]);
        // the block's row maximum of the scores (the scale is positive, so it
        // is applied after the max and folded into the exponent below); a
        // whole block before the pair's first new token needs no mask
        float mx = -INFINITY;
        if (nk == kAttnKeys && k0 + kAttnKeys - 1 <= lim0) {
#pragma unroll
          for (int e = 0; e < kAttnKeys; ++e) mx = fmaxf(mx, sv[e]);
        } else {
#pragma unroll
          for (int e = 0; e < kAttnKeys; ++e) {
            sv[e] = (e < nk && k0 + e <= lim) ? sv[e] : -INFINITY;
            mx = fmaxf(mx, sv[e]);
          }
        }
        mx = row < QRp ? mx * scl : -INFINITY;
        const bool grow = mx > m_run + 8.f;
        float alpha = 1.f;
        if (grow) {
          alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - mx);
          m_run = mx;
        }
        l_run *= alpha;
        // P buffer g & 1 and this warp's O were last used by PV_{g-2}
        if (g >= 2 && !warp_wait(&pv_done[g & 1], ((g >> 1) - 1) & 1, ctx, 85)) {
          dead = true;
          break;
        }
        // this warp's O holds its earlier blocks of the run: rescale it
        const float oa = (grow && j >= 2) ? alpha : 1.f;
        if (__any_sync(0xffffffffu, oa != 1.f)) {
          tc_fence_after();
#pragma unroll 1
          for (int c16 = 0; c16 < 8; ++c16) {
            float ov[16];
            tmem_ld16(t_my + c16 * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= oa;
            tmem_st16(t_my + c16 * 16, ov);
          }
          tmem_wait_st();
        }
        const float nmb = m_run == -INFINITY ? 0.f : -m_run;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[kAttnKeys / 2];
#pragma unroll
        for (int e = 0; e < kAttnKeys; e += 2) {
          const float p0 = ex2_approx(fmaf(sv[e], scl, nmb));
          const float p1 = ex2_approx(fmaf(sv[e + 1], scl, nmb));
          s4[(e >> 1) & 3] += p0 + p1;
          pk[e >> 1] = pack_bf16(p0, p1);
        }
        l_run += (s4[0] + s4[1]) + (s4[2] + s4[3]);
        if (nk < kAttnKeys && quarter == 0) {
          // V rows past the context were not loaded (or are stale)
          uint8_t* vst = attn_v(P, g);
          for (int e = lane; e < (kAttnKeys - nk) * 16; e += 32) {
            const int key = nk + (e >> 4), hf = (e >> 3) & 1, c8 = e & 7;
            *reinterpret_cast<uint4*>(vst + hf * kAttnKeys * 128 + key * 128 + c8 * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        if (row < QRp) {
          uint8_t* prow = ps + (g & 1) * QRp * 128 + row * 128;
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            *reinterpret_cast<uint4*>(prow + ((c8 ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        }
        fence_proxy_async_shared();   // P and the zeroed V rows feed the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[g & 1]);
      }
      // merge the two warps' (max, sum, O) per row: the second hands its max
      // and sum over, the first reads both O and writes Ob and the lse
      if (kk_sm == 1 && row < QRp) {
        row_m1[row] = m_run;
        row_l1[row] = l_run;
      }
      named_bar(3 + quarter, 64);
      if (kk_sm == 0) {
        const float m1 = row < QRp ? row_m1[row] : -INFINITY;
        const float l1 = row < QRp ? row_l1[row] : 0.f;
        const float mm = fmaxf(m_run, m1);
        const float f0 = l_run > 0.f ? exp2f(m_run - mm) : 0.f;
        const float f1 = l1 > 0.f ? exp2f(m1 - mm) : 0.f;
        const float l = l_run * f0 + l1 * f1;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool use0 = __any_sync(0xffffffffu, l_run > 0.f);
        const bool use1 = __any_sync(0xffffffffu, l1 > 0.f);
        bool ok = n > 0 && !dead;
        if (ok) {
          // the last PV into each O
          const int g0 = i + ((n - 1) & ~1);
          const int g1 = i + ((n & 1) ? n - 2 : n - 1);
          ok = warp_wait(&pv_done[g0 & 1], (g0 >> 1) & 1, ctx, 86) &&
               (n < 2 || warp_wait(&pv_done[g1 & 1], (g1 >> 1) & 1, ctx, 87));
          if (!ok) dead = true;
        }
        if (ok) {
          tc_fence_after();
          const uint32_t ta = t_o + static_cast<uint32_t>((i & 1) * 128) + t_lane;
          const uint32_t tb = t_o + static_cast<uint32_t>(((i + 1) & 1) * 128) + t_lane;
#pragma unroll 1
          for (int c16 = 0; c16 < 8; ++c16) {
            float o0[16], o1[16];
            if (use0) tmem_ld16(ta + c16 * 16, o0);
            if (use1) tmem_ld16(tb + c16 * 16, o1);
            tmem_wait_ld();
            if (row < QRp) {
#pragma unroll
              for (int e4 = 0; e4 < 4; ++e4) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int x = e4 * 4 + e;
                  v[e] = ((use0 && l_run > 0.f) ? o0[x] * f0 : 0.f) +
                         ((use1 && l1 > 0.f) ? o1[x] * f1 : 0.f);
                }
                *reinterpret_cast<float4*>(Ob + row * kOP + c16 * 16 + e4 * 4) =
                    make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
              }
            }
          }
          tc_fence_before();
        } else if (row < QRp) {
          for (int e4 = 0; e4 < 32; ++e4)
            *reinterpret_cast<float4*>(Ob + row * kOP + e4 * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (row < QRp) row_lse[row] = l > 0.f ? mm + log2f(l) : -INFINITY;
      }
    }
    if (named_bar_or(1, 256, dead)) return -1;
    attn_pair_out(a, c, u0, p, blk_a, blk_b, Ob, row_lse, pend, &npend);
    named_bar(1, 256);
    i += n;
    u = run_end;
  }
  if (ct == 0) trace_stamp(ctx, c, TR_LOOP_END);
  if (!attn_combine(a, c, ctx, pend, npend, flag, ctb)) return -1;
  if (ct == 0) trace_stamp(ctx, c, TR_END);
  return i;
}

// Consumer side of an attention share (warps 1-8): `priv` is the share's
// private shared memory (layout attn_smem_layout(QRp, 0)).  Returns the
// number of key blocks it consumed (the blocks below each pair's context),
// or -1 after a failed wait.  kU2: two 64-key blocks per iteration below
// 64 query rows (the standalone kernel; the megakernel's register budget,
// shared with its argument copies, keeps one).
template <int kNMT, bool kU2>
__device__ int attn_consume_t(const AttnArgs& a, int c, const Dep& dep,
                              const KernelCtx& ctx, uint8_t* priv, const Pipe& P) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QRp = a.QRp, G = a.Hq / a.Hkv;
  constexpr int nmt = kNMT;
  constexpr int kXS = nmt * 8;   // partial-score floats per thread
  const AttnSmem L = attn_smem_layout(QRp, 0);
  uint8_t* smem = priv;
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem + L.q_off);
  float* Ob = reinterpret_cast<float*>(smem + L.o_off);
  float* xs = reinterpret_cast<float*>(smem + L.xs_off);
  float* kg_m = reinterpret_cast<float*>(smem + L.stat_off);   // [4][QRp]
  float* kg_l = kg_m + 4 * QRp;                                 // [4][QRp]
  float* row_lse = kg_l + 4 * QRp;
  float* row_w = row_lse + QRp;
  int* row_pos = reinterpret_cast<int*>(row_w + QRp);
  int* flag = reinterpret_cast<int*>(smem + L.misc_off);
  int* ctb = flag + 16 + 32 * 4 + 64;     // [kMaxContrib] combine contributors
  const int U = a.R * a.Hkv * a.NB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const Binding* bd = ctx.binding;
  const int ct = tid - 32, wc = warp - 1;  // wc: 0..7
  // Warp wc works on key group kg = wc % 4 (16 keys of every 64-key block).
  // With two 16-row m-tiles (kMS) the pair of a key group splits the query
  // rows: each warp takes one m-tile over the whole head dim, so no partial
  // scores are exchanged; otherwise it splits the head dim (dh), takes every
  // m-tile and the pair exchanges partial scores.
  constexpr bool kMS = (kNMT == 2);
  constexpr int kMT = kMS ? 1 : kNMT;      // m-tiles per warp
  constexpr int kND = kMS ? 16 : 8;        // 8-column d tiles per warp
  constexpr int kU = (kU2 && kNMT < 4) ? 2 : 1;   // 64-key blocks per iteration
  const int kg = wc & 3, dh = wc >> 2;     // key group; d-half or m-tile
  const int mtb = kMS ? dh : 0;            // first m-tile of this warp
  const int dlo = kMS ? 0 : dh;            // first d-half of this warp
  const int partner = kg + 4 * (1 - dh);
  if (ct == 0) {
    trace_stamp(ctx, c, TR_START);
    trace_put(ctx, c, TR_UNITS, static_cast<unsigned long long>(u1 - u0));
  }
  if (!group_wait(dep, ctx, 1, 256, ct == 0, 34, &flag[2])) return -1;
  if (ct == 0) trace_stamp(ctx, c, TR_DEPS);
  const int* pos = resolve<const int>(a.pos, bd);
  const uint16_t* qg = static_cast<const uint16_t*>(a.q);
  const uint32_t qs_u32 = smem_u32(Qs);
  const int qr = lane >> 2, qc = lane & 3;  // fragment row / column pair
  bool dead = false;
  int i = 0;                               // valid-unit counter (matches producer)
  int pend[2], npend = 0;                  // pairs this CTA shares (first / last)
  int u = u0;
  while (u < u1) {
    const int p = static_cast<int>(u / a.NB);
    const int blk_a = static_cast<int>(u % a.NB);
    const int run_end = min(u1, (p + 1) * a.NB);
    const int blk_b = run_end - p * a.NB;
    const int r = p / a.Hkv, h = p % a.Hkv;
    const int ctxr = pos[r * a.T + a.T - 1] + 1;
    // this pair's query rows (swizzled 16-byte chunks) and causal limits
#pragma unroll 4
    for (int e = ct; e < QRp * 16; e += 256) {
      const int rr = e >> 4, ch = e & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (rr < a.QR) {
        const int t = rr / G, g = rr % G;
        const size_t src = (static_cast<size_t>(r * a.T + t) * a.Hq + h * G + g) * 128 + ch * 8;
        v = __ldcg(reinterpret_cast<const uint4*>(qg + src));
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(Qs) + rr * 256 + ((ch ^ (rr & 7)) << 4)) = v;
    }
    for (int rr = ct; rr < QRp; rr += 256) row_pos[rr] = rr < a.QR ? pos[r * a.T + rr / G] : -1;
    named_bar(1, 256);
    int lim[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      lim[mt][0] = row_pos[(mtb + mt) * 16 + qr];
      lim[mt][1] = row_pos[(mtb + mt) * 16 + qr + 8];
    }
    float o[kMT][kND][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int nt = 0; nt < kND; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    float mrow[kMT][2], lrow[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
      mrow[mt][0] = mrow[mt][1] = -INFINITY;
      lrow[mt][0] = lrow[mt][1] = 0.f;
    }
    const int nvb = (ctxr + kAttnKeys - 1) / kAttnKeys;   // valid blocks
    const int blk_end = min(blk_b, nvb);
    // kU blocks per iteration: their scores share one online-softmax update
    // (half the max / sum shuffles and rescales per key) and the two blocks'
    // MMA chains are independent, so each warp has twice the work in flight.
    int it = 0;
    for (int blk = blk_a; blk < blk_end; ++it) {
      const int nu = (kU == 2 && blk + 1 < blk_end) ? 2 : 1;
      if (!dead) dead = !pipe_warp_wait(P, i, ctx, 35);
      if (nu == 2 && !dead) dead = !pipe_warp_wait(P, i + 1, ctx, 35);
      if (i == 0 && ct == 0) trace_stamp(ctx, c, TR_FIRST);
      uint32_t kb_u32[kU], vb_u32[kU];
      int k0[kU], nk[kU];
      bool part = false;
#pragma unroll
      for (int uu = 0; uu < kU; ++uu) {
        const int iu = uu < nu ? i + uu : i;
        kb_u32[uu] = smem_u32(attn_k(P, iu));
        vb_u32[uu] = smem_u32(attn_v(P, iu));
        k0[uu] = (blk + uu) * kAttnKeys;
        nk[uu] = uu < nu ? min(kAttnKeys, ctxr - k0[uu]) : 0;
        if (uu < nu && nk[uu] < kAttnKeys) part = true;
      }
      float sc[kU][kMT][2][4];
#pragma unroll
      for (int uu = 0; uu < kU; ++uu)
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[uu][mt][nt][e] = 0.f;
      if (!dead) {
#pragma unroll
        for (int uu = 0; uu < kU; ++uu) {
          if (uu < nu && nk[uu] < kAttnKeys) {
            // keys past the context were not loaded (or hold stale data):
            // zero this key group's V rows (the pair splits them by d-half)
            // so that 0-probability keys contribute exactly 0
            uint8_t* vh = attn_v(P, i + uu) + dh * kAttnKeys * 128;
            for (int e = lane; e < 16 * 8; e += 32) {
              const int key = kg * 16 + (e >> 3);
              if (key >= nk[uu]) *reinterpret_cast<uint4*>(vh + key * 128 + (e & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        if (part) __syncwarp();
        // S over this warp's d range (both halves with kMS)
#pragma unroll
        for (int dd = 0; dd < (kMS ? 2 : 1); ++dd) {
          const int dhh = dlo + dd;
#pragma unroll
          for (int ks4 = 0; ks4 < 4; ++ks4) {
            uint32_t qa[kMT][4];
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
              const int qrow = (mtb + mt) * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
              const int qch = (dhh * 4 + ks4) * 2 + (lane >> 4);
              ldsm_x4(qs_u32 + qrow * 256 + ((qch ^ (qrow & 7)) << 4), qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3]);
            }
#pragma unroll
            for (int uu = 0; uu < kU; ++uu) {
              if (uu >= nu) break;
              const int key = kg * 16 + (lane & 7) + ((lane >> 4) << 3);
              const int ch = ks4 * 2 + ((lane >> 3) & 1);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(kb_u32[uu] + dhh * kAttnKeys * 128 + key * 128 + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
#pragma unroll
              for (int mt = 0; mt < kMT; ++mt) {
                mma_bf16_16816(sc[uu][mt][0], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], b0, b1);
                mma_bf16_16816(sc[uu][mt][1], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], b2, b3);
              }
            }
          }
        }
        if constexpr (!kMS) {
#pragma unroll
          for (int uu = 0; uu < kU; ++uu) {
            float* mine = xs + ((it & 1) * kU + uu) * (8 * kXS * 32) + wc * (kXS * 32);
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) mine[((mt * 2 + nt) * 4 + e) * 32 + lane] = sc[uu][mt][nt][e];
          }
        }
      }
      // the two d-half warps of this key group exchange partial scores
      // (with kMS: the pair only waits for each other's V zeroing)
      if (!kMS || part) named_bar(2 + kg, 64);
      if (!dead) {
        if constexpr (!kMS) {
#pragma unroll
          for (int uu = 0; uu < kU; ++uu) {
            const float* other = xs + ((it & 1) * kU + uu) * (8 * kXS * 32) + partner * (kXS * 32);
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[uu][mt][nt][e] += other[((mt * 2 + nt) * 4 + e) * 32 + lane];
          }
        }
        // scale, mask, online softmax on this key group's 16 keys of each block
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int uu = 0; uu < kU; ++uu)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int col = kg * 16 + nt * 8 + qc * 2 + e;
                  const int key = k0[uu] + col;
                  const bool valid = col < nk[uu] && key <= lim[mt][hr];
                  const float v = valid ? sc[uu][mt][nt][hr * 2 + e] * a.scale_log2 : -INFINITY;
                  sc[uu][mt][nt][hr * 2 + e] = v;
                  mx = fmaxf(mx, v);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mold = mrow[mt][hr];
            const float mnew = fmaxf(mold, mx);
            const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(mold - mnew);
            float sum = 0.f;
#pragma unroll
            for (int uu = 0; uu < kU; ++uu)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float pv = (mnew == -INFINITY) ? 0.f : exp2f(sc[uu][mt][nt][hr * 2 + e] - mnew);
                  sc[uu][mt][nt][hr * 2 + e] = pv;
                  sum += pv;
                }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            mrow[mt][hr] = mnew;
            lrow[mt][hr] = lrow[mt][hr] * alpha + sum;
            // after the first blocks a row's maximum rarely moves: skip the
            // rescale (a multiply by exactly 1) unless some row of the warp's
            // 8-row group changed
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
              for (int nt = 0; nt < kND; ++nt) {
                o[mt][nt][hr * 2] *= alpha;
                o[mt][nt][hr * 2 + 1] *= alpha;
              }
            }
          }
        }
        // O += P V over this warp's d range (columns [64 dh, 64 dh + 64), or
        // all 128 with kMS)
#pragma unroll
        for (int uu = 0; uu < kU; ++uu) {
          if (uu >= nu) break;
          uint32_t pa[kMT][4];
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt) {
            pa[mt][0] = pack_bf16(sc[uu][mt][0][0], sc[uu][mt][0][1]);
            pa[mt][1] = pack_bf16(sc[uu][mt][0][2], sc[uu][mt][0][3]);
            pa[mt][2] = pack_bf16(sc[uu][mt][1][0], sc[uu][mt][1][1]);
            pa[mt][3] = pack_bf16(sc[uu][mt][1][2], sc[uu][mt][1][3]);
          }
#pragma unroll
          for (int dd = 0; dd < (kMS ? 2 : 1); ++dd) {
            const int dhh = dlo + dd;
#pragma unroll
            for (int cp = 0; cp < 4; ++cp) {        // pairs of 8-column n-tiles
              const int key = kg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
              const int ch = cp * 2 + (lane >> 4);
              uint32_t b0, b1, b2, b3;
              ldsm_x4_t(vb_u32[uu] + dhh * kAttnKeys * 128 + key * 128 + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
#pragma unroll
              for (int mt = 0; mt < kMT; ++mt) {
                mma_bf16_16816(o[mt][dd * 8 + cp * 2], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
                mma_bf16_16816(o[mt][dd * 8 + cp * 2 + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
              }
            }
          }
        }
        if (part) fence_proxy_async_shared();  // zeroed rows vs the next TMA fill
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(pipe_empty(P, pipe_q(P, i)));
          if (nu == 2) mbar_arrive(pipe_empty(P, pipe_q(P, i + 1)));
        }
      }
      blk += nu;
      i += nu;
    }
    // ---- merge the four key groups (fixed order) into Ob, then lse
    if (named_bar_or(1, 256, dead)) return -1;
    if ((kMS || dh == 0) && qc == 0) {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const int r0 = (mtb + mt) * 16 + qr;
        kg_m[kg * QRp + r0] = mrow[mt][0];
        kg_m[kg * QRp + r0 + 8] = mrow[mt][1];
        kg_l[kg * QRp + r0] = lrow[mt][0];
        kg_l[kg * QRp + r0 + 8] = lrow[mt][1];
      }
    }
    named_bar(1, 256);
    for (int rr = ct; rr < QRp; rr += 256) {
      float mx = -INFINITY;
      for (int g4 = 0; g4 < 4; ++g4) mx = fmaxf(mx, kg_m[g4 * QRp + rr]);
      float l = 0.f;
      if (mx != -INFINITY)
        for (int g4 = 0; g4 < 4; ++g4) l += kg_l[g4 * QRp + rr] * exp2f(kg_m[g4 * QRp + rr] - mx);
      row_w[rr] = mx;
      row_lse[rr] = l > 0.f ? mx + log2f(l) : -INFINITY;
      kg_l[rr] = l;   // slot 0 now holds the merged row sum (read after the barrier)
    }
    named_bar(1, 256);
    float fac[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = (mtb + mt) * 16 + qr + hr * 8;
        const float l = kg_l[rr];
        fac[mt][hr] = (l > 0.f && mrow[mt][hr] != -INFINITY) ? exp2f(mrow[mt][hr] - row_w[rr]) / l : 0.f;
      }
    const int col0 = (kMS ? 0 : dh * 64) + qc * 2;
    for (int g4 = 0; g4 < 4; ++g4) {
      if (kg == g4) {
        // per m-tile and 8 d tiles: load the running sum first (no store ->
        // load chains), add this key group's scaled slice, store
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
          for (int n0 = 0; n0 < kND; n0 += 8) {
            float2 prev[2][8];
            if (g4 > 0) {
#pragma unroll
              for (int hr = 0; hr < 2; ++hr)
#pragma unroll
                for (int nt = 0; nt < 8; ++nt)
                  prev[hr][nt] = *reinterpret_cast<const float2*>(
                      Ob + ((mtb + mt) * 16 + qr + hr * 8) * kOP + col0 + (n0 + nt) * 8);
            }
#pragma unroll
            for (int hr = 0; hr < 2; ++hr)
#pragma unroll
              for (int nt = 0; nt < 8; ++nt) {
                float2 v = make_float2(o[mt][n0 + nt][hr * 2] * fac[mt][hr],
                                       o[mt][n0 + nt][hr * 2 + 1] * fac[mt][hr]);
                if (g4 > 0) {
                  v.x += prev[hr][nt].x;
                  v.y += prev[hr][nt].y;
                }
                *reinterpret_cast<float2*>(Ob + ((mtb + mt) * 16 + qr + hr * 8) * kOP + col0 +
                                           (n0 + nt) * 8) = v;
              }
          }
        }
      }
      named_bar(1, 256);
    }
    attn_pair_out(a, c, u0, p, blk_a, blk_b, Ob, row_lse, pend, &npend);
    named_bar(1, 256);
    u = run_end;
  }
  if (ct == 0) trace_stamp(ctx, c, TR_LOOP_END);
  if (!attn_combine(a, c, ctx, pend, npend, flag, ctb)) return -1;
  if (ct == 0) trace_stamp(ctx, c, TR_END);
  return i;
}


// Standalone attention share: the K/V producer (warp 0) and the mma.sync
// consumer, or (kTC) the tcgen05 consumer over `tmem` (512 columns).
template <int kNMT, bool kTC>
__device__ void attn_op_t(const AttnArgs& a, int c, const Dep& dep,
                          const KernelCtx& ctx, uint8_t* smem, uint32_t tmem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QRp = a.QRp;
  const AttnSmem L = kTC ? attn_tc_smem_layout(QRp, a.stages) : attn_smem_layout(QRp, a.stages);
  uint8_t* stage0 = smem + L.stage_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kMaxStages;
  int* flag = reinterpret_cast<int*>(smem + L.misc_off);
  int* pgbuf = flag + 16;                 // [32][4] pages of the producer's batch
  int* ppos = pgbuf + 32 * 4;             // [64] token positions (producer)
  const int S = a.stages;
  const uint32_t smag = fdiv_magic(static_cast<uint32_t>(S));   // S >= 2
  const int U = a.R * a.Hkv * a.NB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const Binding* bd = ctx.binding;
  const CUtensorMap* kvm = &bd->kv_map;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTC ? 1 : 8);   // one MMA commit, or 8 consumer warps
    }
    if (kTC) {
      uint64_t* tb = reinterpret_cast<uint64_t*>(smem + L.tbar_off);
      // split softmax (up to 32 query rows): one warp reads S, four write P
      const bool split = QRp <= 32 && a.split_sm;
      const uint32_t nsm = QRp > 32 ? 2u : 1u;
      mbar_init(&tb[0], 1);                  // s_full: QK^T commit
      mbar_init(&tb[1], 1);
      mbar_init(&tb[2], split ? 1u : nsm);   // s_free: S read from TMEM
      mbar_init(&tb[3], split ? 1u : nsm);
      mbar_init(&tb[4], split ? 4u : nsm);   // p_full: P written
      mbar_init(&tb[5], split ? 4u : nsm);
      mbar_init(&tb[6], 1);                  // pv_done: PV commit
      mbar_init(&tb[7], 1);
      mbar_init(&tb[8], 1);                  // s_ready: S staged (split)
      mbar_init(&tb[9], 1);
      mbar_init(&tb[10], 4);                 // s2_free: staged S read (split)
      mbar_init(&tb[11], 4);
    }
    flag[0] = flag[1] = 0;
    flag[2] = 1;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------ producer (warp 0, lane 0 issues)
    // Blocks that hold none of this step's new keys (the only K/V rows the
    // previous kernel writes) go out before the dependency wait; positions
    // and block table are step inputs.  Lane 0 waits at the first block that
    // holds a new key.
    bool ok = true, deps_ok = false;
    const CUtensorMap* kvm4 = &bd->kv_map4;
    if (lane == 0) {
      fence_tmap_acquire(kvm);
      prefetch_tmap(kvm);
      if (a.kv4) {
        fence_tmap_acquire(kvm4);
        prefetch_tmap(kvm4);
      }
    }
    const int* pos = resolve<const int>(a.pos, bd);
    const int* bt = resolve<const int>(a.bt, bd);
    const int M = a.R * a.T;
    for (int m = lane; m < M; m += 32) {
      // a position outside [0, max_context) is reported; the keys past the
      // plan's blocks are never loaded, so the row is still safe to compute
      const int p = pos[m];
      if (p < 0 || p >= a.max_ctx) report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 33, p);
      ppos[m] = p;
    }
    __syncwarp();
    const uint64_t pol = policy_evict_first();
    const int box = a.P < kAttnKeys ? a.P : kAttnKeys;   // rows per TMA box
    const int npg = kAttnKeys / box;                      // boxes per 64-key unit
    const uint32_t half = kAttnKeys * 128;                // one d-half of K or V
    int i = 0;
    for (int ub = u0; ok && ub < u1; ub += 32) {
      const int nb = min(32, u1 - ub);
      // the batch's page numbers, loaded by the whole warp
      for (int e = lane; e < nb * npg; e += 32) {
        const int j = e / npg, q = e % npg;
        const int u = ub + j;
        const int p = static_cast<int>(u / a.NB), blk = static_cast<int>(u % a.NB);
        const int r = p / a.Hkv;
        const int ctxr = ppos[r * a.T + a.T - 1] + 1;
        const int key = blk * kAttnKeys + q * box;
        const int lp = key / a.P;
        pgbuf[j * 4 + q] = (key < ctxr && lp < a.max_pages)
                               ? bt[static_cast<size_t>(r) * a.max_pages + lp] : -1;
      }
      __syncwarp();
      if (lane == 0) {
        for (int j = 0; j < nb && ok; ++j) {
          const int u = ub + j;
          const int p = static_cast<int>(u / a.NB), blk = static_cast<int>(u % a.NB);
          const int r = p / a.Hkv, h = p % a.Hkv;
          const int ctxr = ppos[r * a.T + a.T - 1] + 1;
          const int k0 = blk * kAttnKeys;
          if (k0 >= ctxr) continue;
          const uint32_t id = fdiv(static_cast<uint32_t>(i), smag);
          const int s = i - static_cast<int>(id) * S;
          if (i >= S && !mbar_wait(&empty[s], (id - 1) & 1, ctx, 31)) {
            ok = false;
            break;
          }
          uint8_t* st = stage0 + s * L.stage_bytes;
          const int nk = min(kAttnKeys, ctxr - k0);
          if (!deps_ok && (k0 + nk > ppos[r * a.T] || (a.pre_stages > 0 && i >= a.pre_stages))) {
            deps_ok = true;
            if (dep.mode == 0) {
              gdc_wait();
              ok = !aborted(ctx.status);
            } else {
              ok = poll_deps(dep, ctx, 30);
            }
            if (!ok) break;
          }
          const int nbox = (nk + box - 1) / box;     // boxes that hold valid keys
          mbar_arrive_expect_tx(&full[s], nbox * box * 128 * 4);
          if (a.kv4) {
            // the whole block in one box: a page holds all 64 keys (one
            // instruction where four took the issuing thread about 0.9 us)
            int page = pgbuf[j * 4];
            if (page < 0 || page >= a.num_pages) {
              report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 32, k0 / a.P);
              page = 0;
            }
            const int rk = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, h, k0 % a.P));
            tma_load_4d(st, kvm4, &full[s], 0, rk, 0, 0, pol);
            ++i;
            continue;
          }
          for (int q = 0; q < nbox; ++q) {
            const int key = k0 + q * box;
            int page = pgbuf[j * 4 + q];
            if (page < 0 || page >= a.num_pages) {
              report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 32, key / a.P);
              page = 0;
            }
            const int rk = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, h, key % a.P));
            const int rv = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 1, h, key % a.P));
            uint8_t* dq = st + q * box * 128;
            tma_load_2d(dq, kvm, &full[s], 0, rk, pol);
            tma_load_2d(dq + half, kvm, &full[s], 64, rk, pol);
            tma_load_2d(dq + 2 * half, kvm, &full[s], 0, rv, pol);
            tma_load_2d(dq + 3 * half, kvm, &full[s], 64, rv, pol);
          }
          ++i;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      i = __shfl_sync(0xffffffffu, i, 0);
      __syncwarp();
    }
    // every thread passes the dependency once (the CTA's completion then
    // implies its dependencies' completion)
    if (dep.mode == 0) {
      gdc_wait();
      gdc_launch_dependents();
    }
    // every K/V load of this share is out: warm L2 with the O projection's
    // first weight tiles (its shares c, c + CTAs, ...)
    if (lane == 0 && ok)
      for (int c2 = c; c2 < a.pf.G; c2 += static_cast<int>(gridDim.x)) prefetch_next_share(a.pf, c2);
    if (lane == 0) {
      const int issued = i;
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / S) * S;
        mbar_drain(&full[s], (last / S) & 1, ctx.budget_ns);
      }
    }
    return;
  }


  Pipe P;
  P.base = stage0;
  P.full = full;
  P.empty = empty;
  P.slot_bytes = static_cast<uint32_t>(L.stage_bytes);
  pipe_set_ns(P, static_cast<uint32_t>(S));
  P.seq0 = 0;
  P.ups = 1;
  P.x_bytes = 0;
  P.empty_cnt = kTC ? 1 : 8;
  if constexpr (kTC)
    attn_consume_tc(a, c, dep, ctx, smem, L, P, tmem);
  else
    attn_consume_t<kNMT, true>(a, c, dep, ctx, smem + S * L.stage_bytes, P);
}

// ========================================================= MEGAKERNEL
// Streaming megakernel: one worker CTA per SM walks its host-built queue of
// instructions.  Its producer warp runs ahead of the consumer warps and
// fills one ring of equal slots in exactly the order the consumers will
// take them, across instruction boundaries: the weights of the next
// projection stream in while the current instruction is still computing,
// fixing up and signalling (the overlap of instruction i + 1's load with
// instruction i's compute on page "Kernel-Mega-PDL", megakernel section).
// Dependent data (activations, KV blocks that hold this step's new keys) is
// issued only after the instruction's event counters are reached.
// GEMM share c: its units fill slots seq, seq + 1, ... (two units per slot
// without gate/up pairing, one otherwise), each unit's activation slice
// after the slot's tiles.  Weights go out as soon as a slot is free;
// activation slices once the share's inputs are ready, and before the
// producer would block on a slot that only the consumption of a pending
// unit can free.  Every armed slot completes even after a failed wait (so
// the ring can be drained).
__device__ __noinline__ bool mk_produce_gemm(const GemmArgs& a_, int c, const Dep& dep_,
                                             const KernelCtx& ctx_, const Pipe& R_, uint32_t seq,
                                             uint32_t* hi) {
  const GemmArgs a = a_;
  const Dep dep = dep_;
  const KernelCtx ctx = ctx_;
  const Pipe R = R_;
  const int npair = a.pair ? 2 : 1;
  const int ups = npair == 1 ? 2 : 1;
  const int U = a.NT * a.KB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const int n = static_cast<int>(u1 - u0);
  const int nslots = (n + ups - 1) / ups;
  const int kel = a.fp8 ? 128 : 64;
  const uint32_t ub = static_cast<uint32_t>(npair * 16384 + a.Mp * 128);
  const int xbytes = ((a.Mp * 128 + 1023) / 1024) * 1024;
  const uint64_t pw = policy_evict_first(), px = policy_evict_last();
  prefetch_tmap(a.tmap_w);
  prefetch_tmap(a.tmap_x);
  bool deps_ok = false, ok = true;
  int pend = 0;    // first unit whose activation slice is not issued yet
  int armed = 0;   // units whose slot is armed
  auto load_x = [&](int i) {
    const int kb = static_cast<int>((u0 + i) % a.KB);
    const uint32_t q = seq + static_cast<uint32_t>(i / ups);
    tma_load_2d(pipe_slot(R, q) + kSlotTiles + (i % ups) * xbytes, a.tmap_x, pipe_full(R, q),
                kb * kel, 0, px);
  };
  for (int j = 0; j < nslots && ok; ++j) {
    const uint32_t q = seq + static_cast<uint32_t>(j);
    if (q >= R.ns) {
      uint64_t* e = pipe_empty(R, q);
      const uint32_t par = (fdiv(q, R.ns_magic) - 1) & 1u;
      if (!deps_ok && pend < armed && !mbar_try_wait(e, par)) {
        deps_ok = poll_deps(dep, ctx, 60);
        trace_stamp(ctx, c, TR_PDEPS);
        for (; pend < armed; ++pend) load_x(pend);
        if (!deps_ok) {
          ok = false;
          break;
        }
      }
      if (!mbar_wait(e, par, ctx, 61)) {
        ok = false;
        break;
      }
    }
    const int i0 = j * ups, i1 = min(n, i0 + ups);
    mbar_arrive_expect_tx(pipe_full(R, q), ub * static_cast<uint32_t>(i1 - i0));
    *hi = q + 1;
    for (int i = i0; i < i1; ++i) {
      const int u = u0 + i;
      const int t = a.t_base + static_cast<int>(u / a.KB), kb = static_cast<int>(u % a.KB);
      tma_load_2d(pipe_slot(R, q) + (i - i0) * 16384, a.tmap_w, pipe_full(R, q), kb * kel,
                  t * 128, pw);
      if (a.pair)
        tma_load_2d(pipe_slot(R, q) + 16384, a.tmap_w, pipe_full(R, q), kb * kel,
                    a.up_row + t * 128, pw);
    }
    armed = i1;
    if (deps_ok)
      for (; pend < armed; ++pend) load_x(pend);
  }
  if (!deps_ok && armed > 0) {
    deps_ok = poll_deps(dep, ctx, 62);
    trace_stamp(ctx, c, TR_PDEPS);
  }
  for (; pend < armed; ++pend) load_x(pend);
  return ok && (deps_ok || armed == 0);
}

// Attention share c (whole warp; lane 0 issues): valid block i (keys below
// its pair's context) takes slot seq + i (K, then V).
// Blocks that hold none of this step's new keys are independent of the
// previous instructions and go out at once; the first block that holds a
// new key waits for the share's inputs.  Returns the valid blocks issued
// (through *nvalid) and false after a failed wait.
__device__ __noinline__ bool mk_produce_attn(const AttnArgs& a_, int c, const Dep& dep_,
                                             const KernelCtx& ctx_, const Pipe& R_, uint32_t seq,
                                             int* pgbuf, int* ppos, int* nvalid, uint32_t* hi) {
  const AttnArgs a = a_;
  const Dep dep = dep_;
  const KernelCtx ctx = ctx_;
  const Pipe R = R_;
  const int lane = threadIdx.x & 31;
  const int U = a.R * a.Hkv * a.NB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const Binding* bd = ctx.binding;
  const CUtensorMap* kvm = &bd->kv_map;
  if (lane == 0) {
    fence_tmap_acquire(kvm);
    prefetch_tmap(kvm);
  }
  const int* pos = resolve<const int>(a.pos, bd);
  const int* bt = resolve<const int>(a.bt, bd);
  const int M = a.R * a.T;
  for (int m = lane; m < M; m += 32) {
    const int p = pos[m];
    if (p < 0 || p >= a.max_ctx) report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 66, p);
    ppos[m] = p;
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();
  const int box = a.P < kAttnKeys ? a.P : kAttnKeys;   // rows per TMA box
  const int npg = kAttnKeys / box;                      // boxes per 64-key block
  const uint32_t half = kAttnKeys * 128;                // one d-half of K or V
  bool ok = true, deps_ok = dep.n == 0;
  int i = 0;
  for (int ub = u0; ok && ub < u1; ub += 32) {
    const int nb = min(32, u1 - ub);
    for (int e = lane; e < nb * npg; e += 32) {
      const int j = e / npg, qq = e % npg;
      const int u = ub + j;
      const int p = static_cast<int>(u / a.NB), blk = static_cast<int>(u % a.NB);
      const int r = p / a.Hkv;
      const int ctxr = ppos[r * a.T + a.T - 1] + 1;
      const int key = blk * kAttnKeys + qq * box;
      const int lp = key / a.P;
      pgbuf[j * 4 + qq] = (key < ctxr && lp < a.max_pages)
                              ? bt[static_cast<size_t>(r) * a.max_pages + lp] : -1;
    }
    __syncwarp();
    if (lane == 0) {
      for (int j = 0; j < nb && ok; ++j) {
        const int u = ub + j;
        const int p = static_cast<int>(u / a.NB), blk = static_cast<int>(u % a.NB);
        const int r = p / a.Hkv, h = p % a.Hkv;
        const int ctxr = ppos[r * a.T + a.T - 1] + 1;
        const int k0 = blk * kAttnKeys;
        if (k0 >= ctxr) continue;
        const int nk = min(kAttnKeys, ctxr - k0);
        if (!deps_ok && k0 + nk > ppos[r * a.T]) {
          deps_ok = poll_deps(dep, ctx, 63);
          trace_stamp(ctx, c, TR_PDEPS);
          if (!deps_ok) {
            ok = false;
            break;
          }
        }
        const int nbox = (nk + box - 1) / box;
        const uint32_t q = seq + static_cast<uint32_t>(i);
        if (q >= R.ns && !mbar_wait(pipe_empty(R, q), (fdiv(q, R.ns_magic) - 1) & 1u, ctx, 64)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(pipe_full(R, q), static_cast<uint32_t>(nbox * box * 128 * 4));
        *hi = q + 1;
        uint8_t* dst = pipe_slot(R, q);
        for (int qq = 0; qq < nbox; ++qq) {
          const int key = k0 + qq * box;
          int page = pgbuf[j * 4 + qq];
          if (page < 0 || page >= a.num_pages) {
            report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 65, key / a.P);
            page = 0;
          }
          const int rk = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, h, key % a.P));
          const int rv = static_cast<int>(kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 1, h, key % a.P));
          uint8_t* dq = dst + qq * box * 128;
          tma_load_2d(dq, kvm, pipe_full(R, q), 0, rk, pol);
          tma_load_2d(dq + half, kvm, pipe_full(R, q), 64, rk, pol);
          tma_load_2d(dq + 2 * half, kvm, pipe_full(R, q), 0, rv, pol);
          tma_load_2d(dq + 3 * half, kvm, pipe_full(R, q), 64, rv, pol);
        }
        ++i;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    i = __shfl_sync(0xffffffffu, i, 0);
    deps_ok = __shfl_sync(0xffffffffu, deps_ok ? 1 : 0, 0) != 0;
    __syncwarp();
  }
  *nvalid = i;
  return ok;
}

// Consumer side of one GEMM instruction with the variant its arguments call
// for, over the worker's ring and TMEM accumulator ring.
// Each consumer variant is a separate, non-inlined function (the megakernel
// then allocates registers per variant, as the standalone kernels do, not
// for the union of all of them), and it works on private copies of its
// arguments: the instruction's arguments sit in shared memory and the
// descriptors in the caller's frame, and every inline-asm memory clobber
// (barrier waits, MMAs, fences) would otherwise force the compiler to load
// each field again; the standalone kernels read them from parameter space,
// which never changes.
template <int kMG, int kMp>
__device__ __noinline__ void mk_gemm_v(const GemmArgs& a_, int c, const Dep& dep_,
                                       const KernelCtx& ctx_, const GemmShared& sh_,
                                       const Pipe& P_, const TmemRing& TR_) {
  const GemmArgs a = a_;
  const Dep dep = dep_;
  const KernelCtx ctx = ctx_;
  const GemmShared sh = sh_;
  const Pipe P = P_;
  const TmemRing TR = TR_;
  gemm_consume_t<kMG, kMp, false>(a, c, dep, ctx, sh, P, TR);
}

template <int kNMT>
__device__ __noinline__ int mk_attn_v(const AttnArgs& a_, int c, const Dep& dep_,
                                      const KernelCtx& ctx_, uint8_t* priv, const Pipe& P_) {
  const AttnArgs a = a_;
  const Dep dep = dep_;
  const KernelCtx ctx = ctx_;
  const Pipe P = P_;
  return attn_consume_t<kNMT, false>(a, c, dep, ctx, priv, P);
}

__device__ __noinline__ void mk_norm(const NormArgs& a_, int c, const Dep& dep_,
                                     const KernelCtx& ctx_, uint8_t* priv) {
  const NormArgs a = a_;
  const Dep dep = dep_;
  const KernelCtx ctx = ctx_;
  // one engine for every H (the megakernel's code stays small), without
  // the deferred fix-up's partial sums (its projections finish their tiles)
  norm_op<4, false>(a, c, dep, ctx, priv);
}

__device__ void mk_gemm(const GemmArgs& a, int c, const Dep& dep, const KernelCtx& ctx,
                        uint8_t* priv, const Pipe& P, const TmemRing& TR, uint64_t* tbars) {
  GemmShared sh = gemm_shared(a, priv, 0);
  sh.tfull = tbars;            // [4]
  sh.tempty = tbars + 4;       // [4]
  sh.tready = tbars + 8;       // [2]
  sh.tfree = tbars + 10;       // [2]
  sh.tprep = nullptr;          // the epilogue warps stage the QKV operands
  if (!a.mma) {
    if (a.M <= 1)
      mk_gemm_v<1, 0>(a, c, dep, ctx, sh, P, TR);
    else if (a.M <= 2)
      mk_gemm_v<2, 0>(a, c, dep, ctx, sh, P, TR);
    else
      mk_gemm_v<4, 0>(a, c, dep, ctx, sh, P, TR);
  } else {
    if (a.Mp <= 16)
      mk_gemm_v<0, 16>(a, c, dep, ctx, sh, P, TR);
    else if (a.Mp <= 32)
      mk_gemm_v<0, 32>(a, c, dep, ctx, sh, P, TR);
    else
      mk_gemm_v<0, 64>(a, c, dep, ctx, sh, P, TR);
  }
}

// Consumer side of one attention instruction; returns the key blocks it
// consumed, or -1 after a failed wait.
__device__ int mk_attn(const AttnArgs& a, int c, const Dep& dep, const KernelCtx& ctx,
                       uint8_t* priv, const Pipe& P) {
  if (a.QRp <= 16) return mk_attn_v<1>(a, c, dep, ctx, priv, P);
  if (a.QRp <= 32) return mk_attn_v<2>(a, c, dep, ctx, priv, P);
  return mk_attn_v<4>(a, c, dep, ctx, priv, P);
}

// Units of GEMM share c (its Stream-K range).
__device__ __forceinline__ int gemm_share_units(const GemmArgs& a, int c) {
  const int U = a.NT * a.KB;
  return static_cast<int>(sk_begin(U, a.G, c + 1) - sk_begin(U, a.G, c));
}

// Tiles GEMM share c hands to its fix-up warps: every tile its range
// touches but the last (which the epilogue warps finish themselves).
__device__ __forceinline__ int gemm_share_handoffs(const GemmArgs& a, int c) {
  const int U = a.NT * a.KB;
  const int u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  return u1 > u0 ? static_cast<int>((u1 - 1) / a.KB - u0 / a.KB) : 0;
}

}  // namespace dl
