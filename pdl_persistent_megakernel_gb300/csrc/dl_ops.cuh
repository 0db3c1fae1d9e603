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
__device__ __forceinline__ long long sk_begin(long long U, int G, int c) {
  return (U * c) / G;
}

// The CTA whose range holds unit x (the last CTA whose range starts <= x).
__device__ __forceinline__ int sk_owner(long long U, int G, long long x) {
  int c = static_cast<int>((x * G) / U);
  if (c >= G) c = G - 1;
  while (c > 0 && sk_begin(U, G, c) > x) --c;
  while (c + 1 < G && sk_begin(U, G, c + 1) <= x) ++c;
  return c;
}

// =================================================================== NORM
// Residual add + RMSNorm (+ per-token, per-128-group e4m3 quantisation):
//   r = bf16(x + res);  h = r * rsqrt(mean(r^2) + eps) * w
// One CTA handles rows [c * rows_per_cta, ...); 256 consumer threads, 16-byte
// vectors, H <= 8192.
__device__ void norm_op(const NormArgs& a, int c, const Dep& dep,
                        const KernelCtx& ctx, uint8_t* smem) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    idle_wait(dep);
    return;
  }
  const int ct = tid - 32, lane = tid & 31, wc = ct >> 5;
  float* red = reinterpret_cast<float*>(smem);     // [2][8]
  int* sflag = reinterpret_cast<int*>(smem + 128);
  if (!group_wait(dep, ctx, 1, 256, ct == 0, 1, sflag)) return;
  const Binding* bd = ctx.binding;
  const uint16_t* x = resolve<const uint16_t>(a.x, bd);
  const uint16_t* res = resolve<const uint16_t>(a.res, bd);
  uint16_t* rout = resolve<uint16_t>(a.r_out, bd);
  const uint16_t* w = static_cast<const uint16_t*>(a.w);
  const int H = a.H, nvec = H >> 3;
  const int m0 = c * a.rows_per_cta;
  const int m1 = min(a.M, m0 + a.rows_per_cta);
  for (int m = m0; m < m1; ++m) {
    float r[4][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = ct + j * 256;
      if (v < nvec) {
        const size_t off = static_cast<size_t>(m) * H + v * 8;
        const uint4 xv = __ldcg(reinterpret_cast<const uint4*>(x + off));
        const uint4 rv = __ldcg(reinterpret_cast<const uint4*>(res + off));
        const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t rs[4] = {rv.x, rv.y, rv.z, rv.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = bfround(bf16_lo(xs[e]) + bf16_lo(rs[e]));
          const float a1 = bfround(bf16_hi(xs[e]) + bf16_hi(rs[e]));
          r[j][2 * e] = a0;
          r[j][2 * e + 1] = a1;
          ss += a0 * a0 + a1 * a1;
          o[e] = static_cast<uint32_t>(f2bf(a0)) |
                 (static_cast<uint32_t>(f2bf(a1)) << 16);
        }
        *reinterpret_cast<uint4*>(rout + off) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) red[(m & 1) * 8 + wc] = ss;
    named_bar(1, 256);
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += red[(m & 1) * 8 + i];
    const float inv = rsqrtf(tot / static_cast<float>(H) + a.eps);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = ct + j * 256;
      const bool act = v < nvec;
      float h[8];
      if (act) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(w + v * 8));
        const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[2 * e] = r[j][2 * e] * inv * bf16_lo(ws[e]);
          h[2 * e + 1] = r[j][2 * e + 1] * inv * bf16_hi(ws[e]);
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
}

// =================================================================== GEMM
struct GemmSmem {
  int w_bytes, x_bytes, stage_bytes, tile_off, bar_off, misc_off, nb_off, total;
};

__host__ __device__ inline GemmSmem gemm_smem_layout(int npair, int Mp,
                                                     int stages) {
  GemmSmem L;
  L.w_bytes = 16384;
  L.x_bytes = ((Mp * 128 + 1023) / 1024) * 1024;
  L.stage_bytes = npair * L.w_bytes + L.x_bytes;
  L.tile_off = stages * L.stage_bytes;
  L.bar_off = L.tile_off + npair * Mp * 128 * 4;
  L.misc_off = L.bar_off + (2 * kMaxStages + 4) * 8;  // flags, reductions
  L.nb_off = L.misc_off + 256;                         // rope exchange [4][128]
  L.total = L.nb_off + 4 * 128 * 4;
  return L;
}

struct GemmShared {
  uint8_t* stage0;
  float* tout;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  int* flag;      // [4]
  float* red;     // [2][2][4] reductions
  float* nb;      // [2][128] rope exchange (aliases misc space below)
  int* bidx;      // [2][4]
};

// ------------------------------------------------------- GEMM epilogues
// tout = the finished tile: [npair][Mp][128] fp32 (rows of the weight tile on
// the fast axis).  nthr threads (128 or 256) with group barrier `bar`;
// tokens are processed by groups of 128 threads.

__device__ void epi_store_bf16(const GemmArgs& a, int tg, const float* tout,
                               int nthr, int ct, const Binding* bd) {
  uint16_t* out = resolve<uint16_t>(a.out, bd);
  for (int e = ct; e < a.M * 128; e += nthr) {
    const int m = e >> 7, i = e & 127;
    out[static_cast<size_t>(m) * a.ldo + tg * 128 + i] = f2bf(tout[m * 128 + i]);
  }
}

__device__ void epi_qkv_rope(const GemmArgs& a, int tg, const float* tout,
                             int nthr, int ct, int bar, const KernelCtx& ctx,
                             const GemmShared& sh) {
  const int ng = nthr >> 7, g = ct >> 7, i = ct & 127, wg = (ct >> 5) & 3;
  const int lane = ct & 31;
  const Binding* bd = ctx.binding;
  const int* pos = resolve<const int>(a.pos, bd);
  const int* bt = resolve<const int>(a.bt, bd);
  uint16_t* kv = resolve<uint16_t>(a.kv, bd);
  const int hh = tg;
  const bool is_q = hh < a.Hq;
  const bool is_k = !is_q && hh < a.Hq + a.Hkv;
  float wn = 1.f;
  if (is_q || is_k) {
    const uint16_t* nw = static_cast<const uint16_t*>(is_q ? a.q_norm_w : a.k_norm_w);
    wn = __uint_as_float(static_cast<uint32_t>(nw[i]) << 16);
  }
  for (int mb = 0; mb < a.M; mb += ng) {
    const int m = mb + g;
    const bool act = m < a.M;
    const float v = act ? bfround(tout[m * 128 + i]) : 0.f;
    float outv = v;
    int p = 0;
    if (act) {
      p = pos[m];
      if (p < 0 || p >= a.rope_max_pos) {
        report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 20, p);
        p = 0;
      }
    }
    if (is_q || is_k) {
      const float ss = warp_sum(v * v);
      if (lane == 0) sh.red[((mb / ng) & 1) * 8 + g * 4 + wg] = ss;
      named_bar(bar, nthr);
      const float* rr = sh.red + ((mb / ng) & 1) * 8 + g * 4;
      const float tot = rr[0] + rr[1] + rr[2] + rr[3];
      const float xn = bfround(v * rsqrtf(tot * (1.f / 128.f) + a.eps) * wn);
      sh.nb[(((mb / ng) & 1) * 2 + g) * 128 + i] = xn;
      named_bar(bar, nthr);
      const float partner = sh.nb[(((mb / ng) & 1) * 2 + g) * 128 + (i ^ 64)];
      const float2 cs = *reinterpret_cast<const float2*>(
          a.rope_cs + (static_cast<size_t>(p) * 64 + (i & 63)) * 2);
      outv = i < 64 ? xn * cs.x - partner * cs.y : xn * cs.x + partner * cs.y;
    }
    if (!act) continue;
    const uint16_t ob = f2bf(outv);
    if (is_q) {
      static_cast<uint16_t*>(a.q_out)[(static_cast<size_t>(m) * a.Hq + hh) * 128 + i] = ob;
    } else {
      const int kvsel = is_k ? 0 : 1;
      const int kh = is_k ? hh - a.Hq : hh - a.Hq - a.Hkv;
      const int r = m / a.T;
      const int lp = p / a.P;
      const int page = lp < a.max_pages ? bt[static_cast<size_t>(r) * a.max_pages + lp] : -1;
      if (page < 0 || page >= a.num_pages) {
        report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 21, lp);
        continue;
      }
      const size_t off =
          kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, kvsel, kh, p % a.P) * 128 + i;
      kv[off] = ob;
    }
  }
}

__device__ void epi_silu_mul(const GemmArgs& a, int tg, const float* tout,
                             int nthr, int ct, int bar, const GemmShared& sh) {
  const int ng = nthr >> 7, g = ct >> 7, i = ct & 127, wg = (ct >> 5) & 3;
  const int lane = ct & 31;
  for (int mb = 0; mb < a.M; mb += ng) {
    const int m = mb + g;
    const bool act = m < a.M;
    float av = 0.f;
    if (act) {
      const float gv = bfround(tout[m * 128 + i]);
      const float uv = bfround(tout[(a.Mp + m) * 128 + i]);
      av = gv / (1.f + expf(-gv)) * uv;
    }
    if (!a.fp8) {
      if (act)
        static_cast<uint16_t*>(a.act)[static_cast<size_t>(m) * a.act_ld + tg * 128 + i] = f2bf(av);
    } else {
      const float am = warp_max(fabsf(av));
      if (lane == 0) sh.red[((mb / ng) & 1) * 8 + g * 4 + wg] = am;
      named_bar(bar, nthr);
      const float* rr = sh.red + ((mb / ng) & 1) * 8 + g * 4;
      const float amax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
      const float s = amax > 0.f ? amax / 448.f : 1.f;
      if (act) {
        static_cast<uint8_t*>(a.act)[static_cast<size_t>(m) * a.act_ld + tg * 128 + i] = f2e4m3(av / s);
        if (i == 0) a.act_scale[static_cast<size_t>(m) * (a.act_ld >> 7) + tg] = s;
      }
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
  const int ng = nthr >> 7, g = ct >> 7, i = ct & 127, wg = (ct >> 5) & 3;
  const int lane = ct & 31;
  for (int mb = 0; mb < a.M; mb += ng) {
    const int m = mb + g;
    const bool act = m < a.M;
    float v = act ? tout[m * 128 + i] : -INFINITY;
    int idx = tg * 128 + i;
    if (act) logits[static_cast<size_t>(m) * a.ldo + idx] = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov > v || (ov == v && oi < idx)) {
        v = ov;
        idx = oi;
      }
    }
    if (lane == 0) {
      sh.red[((mb / ng) & 1) * 8 + g * 4 + wg] = v;
      sh.bidx[((mb / ng) & 1) * 8 + g * 4 + wg] = idx;
    }
    named_bar(bar, nthr);
    if (act && i == 0) {
      const float* rv = sh.red + ((mb / ng) & 1) * 8 + g * 4;
      const int* ri = sh.bidx + ((mb / ng) & 1) * 8 + g * 4;
      float bv = rv[0];
      int bi = ri[0];
      for (int k = 1; k < 4; ++k)
        if (rv[k] > bv || (rv[k] == bv && ri[k] < bi)) {
          bv = rv[k];
          bi = ri[k];
        }
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
  // one warp per token
  const int wn = nthr >> 5, wi = ct >> 5;
  for (int m = wi; m < a.M; m += wn) {
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
__device__ void gemm_finish_tile(const GemmArgs& a, int c, long long u0, int tl,
                                 bool full_tile, int npair, int nthr, int ct,
                                 int bar, const KernelCtx& ctx,
                                 const GemmShared& sh) {
  float* tout = sh.tout;
  const int nel = npair * a.Mp * 128;
  if (!full_tile) {
    const long long U = static_cast<long long>(a.NT) * a.KB;
    const long long ts = static_cast<long long>(tl) * a.KB;
    const int slot = (u0 >= ts) ? 0 : 1;
    float* mine = a.ws + static_cast<size_t>(c * 2 + slot) * nel;
    for (int e = ct; e < nel; e += nthr) mine[e] = tout[e];
    __threadfence();
    named_bar(bar, nthr);
    const int cf = sk_owner(U, a.G, ts);
    const int cl = sk_owner(U, a.G, ts + a.KB - 1);
    if (ct == 0) {
      int n = 0;
      for (int cc = cf; cc <= cl; ++cc)
        if (sk_begin(U, a.G, cc + 1) > sk_begin(U, a.G, cc)) ++n;
      const unsigned old = atomicAdd(a.tile_cnt + tl, 1u);
      sh.flag[0] = (old + 1 == static_cast<unsigned>(n)) ? 1 : 0;
    }
    named_bar(bar, nthr);
    if (!sh.flag[0]) return;
    __threadfence();
    for (int e = ct; e < nel; e += nthr) {
      float s = 0.f;
      for (int cc = cf; cc <= cl; ++cc) {
        const long long b0 = sk_begin(U, a.G, cc);
        if (sk_begin(U, a.G, cc + 1) <= b0) continue;
        if (cc == c) {
          s += tout[e];
        } else {
          const int sl = (b0 >= ts) ? 0 : 1;
          s += __ldcg(a.ws + static_cast<size_t>(cc * 2 + sl) * nel + e);
        }
      }
      tout[e] = s;
    }
    if (ct == 0) a.tile_cnt[tl] = 0u;
    named_bar(bar, nthr);
  }
  const int tg = a.t_base + tl;
  switch (a.epi) {
    case EPI_QKV_ROPE:
      epi_qkv_rope(a, tg, tout, nthr, ct, bar, ctx, sh);
      break;
    case EPI_STORE_BF16:
      epi_store_bf16(a, tg, tout, nthr, ct, ctx.binding);
      break;
    case EPI_SILU_MUL:
      epi_silu_mul(a, tg, tout, nthr, ct, bar, sh);
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

// ------------------------------------------------------------ GEMM engine
// kMG: GEMV token bound (1/2/4/8, CUDA cores); kMp: tcgen05 N (16/32/64).
// Exactly one of them is non-zero.
template <int kMG, int kMp>
__device__ void gemm_op_t(const GemmArgs& a, int c, const Dep& dep,
                          const KernelCtx& ctx, uint8_t* smem,
                          uint32_t tmem_base) {
  constexpr bool kMMA = kMp > 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int npair = a.pair ? 2 : 1;
  const GemmSmem L = gemm_smem_layout(npair, a.Mp, a.stages);
  GemmShared sh;
  sh.stage0 = smem;
  sh.tout = reinterpret_cast<float*>(smem + L.tile_off);
  sh.full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  sh.empty = sh.full + kMaxStages;
  sh.tfull = sh.empty + kMaxStages;
  sh.tempty = sh.tfull + 2;
  sh.flag = reinterpret_cast<int*>(smem + L.misc_off);
  sh.red = reinterpret_cast<float*>(smem + L.misc_off + 16);
  sh.bidx = reinterpret_cast<int*>(smem + L.misc_off + 16 + 64);
  sh.nb = reinterpret_cast<float*>(smem + L.nb_off);
  const long long U = static_cast<long long>(a.NT) * a.KB;
  const long long u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  const int nunits = static_cast<int>(u1 - u0);
  const int S = a.stages;
  const int kel = a.fp8 ? 128 : 64;  // elements per k-block
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kMMA ? 1 : 8);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.tfull[b], 1);
      mbar_init(&sh.tempty[b], 4);
    }
    sh.flag[0] = sh.flag[1] = 0;
    sh.flag[2] = 1;
    sh.flag[3] = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------- producer
    if (lane != 0) {
      idle_wait(dep);
      return;
    }
    prefetch_tmap(a.tmap_w);
    prefetch_tmap(a.tmap_x);
    const uint32_t tx = npair * 16384 + a.Mp * 128;
    const uint64_t pw = policy_evict_first(), px = policy_evict_last();
    const int pre = min(S, nunits);
    // weights of the first stages do not depend on the previous op
    for (int i = 0; i < pre; ++i) {
      const long long u = u0 + i;
      const int t = a.t_base + static_cast<int>(u / a.KB), kb = static_cast<int>(u % a.KB);
      uint8_t* st = sh.stage0 + i * L.stage_bytes;
      mbar_arrive_expect_tx(&sh.full[i], tx);
      tma_load_2d(st, a.tmap_w, &sh.full[i], kb * kel, t * 128, pw);
      if (a.pair)
        tma_load_2d(st + 16384, a.tmap_w, &sh.full[i], kb * kel, a.up_row + t * 128, pw);
    }
    bool ok = single_wait(dep, ctx, 10);
    // activations of the prefetched stages (issued even after a failed wait
    // so that every armed stage completes and can be drained)
    for (int i = 0; i < pre; ++i) {
      const int kb = static_cast<int>((u0 + i) % a.KB);
      tma_load_2d(sh.stage0 + i * L.stage_bytes + npair * 16384, a.tmap_x, &sh.full[i],
                  kb * kel, 0, px);
    }
    int issued = pre;
    if (ok) {
      for (int i = pre; i < nunits; ++i) {
        const int s = i % S;
        if (!mbar_wait(&sh.empty[s], ((i / S) - 1) & 1, ctx, 11)) break;
        const long long u = u0 + i;
        const int t = a.t_base + static_cast<int>(u / a.KB), kb = static_cast<int>(u % a.KB);
        uint8_t* st = sh.stage0 + s * L.stage_bytes;
        mbar_arrive_expect_tx(&sh.full[s], tx);
        tma_load_2d(st, a.tmap_w, &sh.full[s], kb * kel, t * 128, pw);
        if (a.pair)
          tma_load_2d(st + 16384, a.tmap_w, &sh.full[s], kb * kel, a.up_row + t * 128, pw);
        tma_load_2d(st + npair * 16384, a.tmap_x, &sh.full[s], kb * kel, 0, px);
        issued = i + 1;
      }
    }
    // no copy may be in flight when the CTA leaves
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / S) * S;  // last unit issued to stage s
      mbar_drain(&sh.full[s], (last / S) & 1, ctx.budget_ns);
    }
    return;
  }

  if constexpr (!kMMA) {
    // ----------------------------------------------- CUDA-core GEMV (M <= 8)
    const int ct = tid - 32;
    if (!group_wait(dep, ctx, 1, 256, ct == 0, 12, &sh.flag[2])) return;
    const int c8 = ct & 7, r0 = ct >> 3;
    int i = 0;
    while (i < nunits) {
      const long long u = u0 + i;
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
        const int s = i % S;
        if (ct == 0) sh.flag[2] = mbar_wait(&sh.full[s], (i / S) & 1, ctx, 13) ? 1 : 0;
        named_bar(1, 256);
        if (!sh.flag[2]) return;
        const uint8_t* st = sh.stage0 + s * L.stage_bytes;
        const uint8_t* xs = st + npair * 16384;
        uint4 xv[kMG];
#pragma unroll
        for (int m = 0; m < kMG; ++m)
          xv[m] = *reinterpret_cast<const uint4*>(xs + m * 128 + ((c8 ^ (m & 7)) << 4));
        const int kb = kb0 + k;
        const int tg = a.t_base + tl;
        for (int p = 0; p < npair; ++p) {
          float sw = 1.f;
          if (a.fp8) {
            const int rt = p == 0 ? tg : (a.up_row >> 7) + tg;
            sw = __ldg(a.w_scale + static_cast<size_t>(rt) * a.KB + kb);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = r0 + 32 * j;
            const uint4 wv = *reinterpret_cast<const uint4*>(
                st + p * 16384 + r * 128 + ((c8 ^ (r & 7)) << 4));
            if (!a.fp8) {
#pragma unroll
              for (int m = 0; m < kMG; ++m) acc[p][j][m] += dot8_bf16(wv, xv[m]);
            } else {
              float wf[16];
              unpack_e4m3x16(wv, wf);
#pragma unroll
              for (int m = 0; m < kMG; ++m) {
                float xf[16];
                unpack_e4m3x16(xv[m], xf);
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) d = fmaf(wf[e], xf[e], d);
                const float sa = m < a.M ? __ldcg(a.x_scale + static_cast<size_t>(m) * a.KB + kb) : 0.f;
                acc[p][j][m] = fmaf(d, sw * sa, acc[p][j][m]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[s]);
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
      named_bar(1, 256);
      gemm_finish_tile(a, c, u0, tl, kb0 == 0 && run == a.KB, npair, 256, ct, 1, ctx, sh);
    }
  } else {
    // --------------------------------------------- tcgen05 (M > 8, N = kMp)
    const int ncols = npair * kMp;  // TMEM columns per accumulator buffer
    if (warp == 1) {
      idle_wait(dep);
      if (lane == 0) {
        const uint32_t idesc = umma_idesc(kMp, !a.fp8);
        int issued = 0;
        for (int i = 0; i < nunits; ++i) {
          const int s = i % S, b = i & 1;
          if (!mbar_wait(&sh.full[s], (i / S) & 1, ctx, 14)) break;
          if (i >= 2 && !mbar_wait(&sh.tempty[b], ((i >> 1) - 1) & 1, ctx, 15)) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(sh.stage0 + s * L.stage_bytes);
          for (int p = 0; p < npair; ++p) {
            const uint32_t d = tmem_base + b * ncols + p * kMp;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = umma_desc_sw128(sa + p * 16384 + k * 32);
              const uint64_t bd = umma_desc_sw128(sa + npair * 16384 + k * 32);
              if (a.fp8)
                umma_e4m3(d, ad, bd, idesc, k > 0 ? 1u : 0u);
              else
                umma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
          }
          umma_commit(&sh.empty[s]);
          umma_commit(&sh.tfull[b]);
          issued = i + 1;
        }
        // no MMA may still read shared memory or write TMEM when we leave
        if (issued > 0)
          mbar_drain(&sh.tfull[(issued - 1) & 1], ((issued - 1) >> 1) & 1, ctx.budget_ns);
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
    if (!group_wait(dep, ctx, 2, 128, et == 0, 16, &sh.flag[2])) return;
    int i = 0;
    while (i < nunits) {
      const long long u = u0 + i;
      const int tl = static_cast<int>(u / a.KB), kb0 = static_cast<int>(u % a.KB);
      const int run = min(nunits - i, a.KB - kb0);
      const int tg = a.t_base + tl;
      float acc[2][kMp];
#pragma unroll
      for (int p = 0; p < 2; ++p)
#pragma unroll
        for (int m = 0; m < kMp; ++m) acc[p][m] = 0.f;
      for (int k = 0; k < run; ++k, ++i) {
        const int b = i & 1;
        if (et == 0) sh.flag[2] = mbar_wait(&sh.tfull[b], (i >> 1) & 1, ctx, 17) ? 1 : 0;
        named_bar(2, 128);
        if (!sh.flag[2]) return;
        tc_fence_after();
        const int kb = kb0 + k;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          if (p >= npair) break;
          float sw = 1.f;
          if (a.fp8) {
            const int rt = p == 0 ? tg : (a.up_row >> 7) + tg;
            sw = __ldg(a.w_scale + static_cast<size_t>(rt) * a.KB + kb);
          }
#pragma unroll
          for (int c16 = 0; c16 < kMp / 16; ++c16) {
            float v[16];
            tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * ncols + p * kMp + c16 * 16, v);
            tmem_wait_ld();
            if (a.fp8) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int m = c16 * 16 + e;
                const float sa = m < a.M ? __ldcg(a.x_scale + static_cast<size_t>(m) * a.KB + kb) : 0.f;
                acc[p][m] = fmaf(v[e], sw * sa, acc[p][m]);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[p][c16 * 16 + e] += v[e];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.tempty[b]);
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        if (p >= npair) break;
#pragma unroll
        for (int m = 0; m < kMp; ++m)
          if (m < a.M) sh.tout[(p * a.Mp + m) * 128 + row] = acc[p][m];
      }
      named_bar(2, 128);
      gemm_finish_tile(a, c, u0, tl, kb0 == 0 && run == a.KB, npair, 128, et, 2, ctx, sh);
    }
  }
}

// ============================================================== ATTENTION
struct AttnSmem {
  int stage_bytes, q_off, s_off, p_off, o_off, stat_off, bar_off, misc_off, total;
};

constexpr int kSPitch = 68;   // fp32 score row pitch (64 keys + pad)

__host__ __device__ inline AttnSmem attn_smem_layout(int QRp, int stages) {
  AttnSmem L;
  L.stage_bytes = 2 * kAttnKeys * 128 * 2;            // K + V, 64 keys x 128 d bf16
  L.q_off = stages * L.stage_bytes;                   // bf16 [QRp][128], swizzled
  L.s_off = L.q_off + QRp * 256;                      // fp32 [QRp][kSPitch]
  L.p_off = L.s_off + QRp * kSPitch * 4;              // bf16 [QRp][64], swizzled
  L.o_off = L.p_off + QRp * 128;                      // fp32 [QRp][128]
  L.stat_off = L.o_off + QRp * 128 * 4;               // m, l, scale, lse, wsum [QRp] + pos
  L.bar_off = L.stat_off + QRp * 4 * 6 + 64;
  L.bar_off = (L.bar_off + 15) & ~15;
  L.misc_off = L.bar_off + 2 * kMaxStages * 8;
  L.total = L.misc_off + 64;
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

// Split-KV GQA decode attention over 64-key blocks with an online softmax
// (base-2 exponentials, scores pre-scaled by log2(e)/sqrt(d)), partial
// outputs normalised per split with their log-sum-exp, and the combine
//   lse = log sum_i e^{lse_i},  O = sum_i e^{lse_i - lse} O_i
// done by the last CTA of each (request, kv head) pair.  QR = T*G query rows
// share one K/V stream; row rr = t*G + g is token r*T + t, q head h*G + g,
// causal limit positions[r*T + t].
__device__ void attn_op(const AttnArgs& a, int c, const Dep& dep,
                        const KernelCtx& ctx, uint8_t* smem) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int QRp = a.QRp, nmt = QRp >> 4, G = a.Hq / a.Hkv;
  const AttnSmem L = attn_smem_layout(QRp, a.stages);
  uint8_t* stage0 = smem;
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem + L.q_off);
  float* Sb = reinterpret_cast<float*>(smem + L.s_off);
  uint16_t* Pb = reinterpret_cast<uint16_t*>(smem + L.p_off);
  float* Ob = reinterpret_cast<float*>(smem + L.o_off);
  float* row_m = reinterpret_cast<float*>(smem + L.stat_off);
  float* row_l = row_m + QRp;
  float* row_sc = row_l + QRp;
  float* row_lse = row_sc + QRp;
  float* row_w = row_lse + QRp;
  int* row_pos = reinterpret_cast<int*>(row_w + QRp);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint64_t* empty = full + kMaxStages;
  int* flag = reinterpret_cast<int*>(smem + L.misc_off);
  const int S = a.stages;
  const long long U = static_cast<long long>(a.R) * a.Hkv * a.NB;
  const long long u0 = sk_begin(U, a.G, c), u1 = sk_begin(U, a.G, c + 1);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    flag[0] = flag[1] = 0;
    flag[2] = 1;
    fence_barrier_init();
  }
  __syncthreads();
  const Binding* bd = ctx.binding;

  if (warp == 0) {
    if (lane != 0) {
      idle_wait(dep);
      return;
    }
    // ------------------------------------------------------- producer
    bool ok = single_wait(dep, ctx, 30);
    const int* pos = resolve<const int>(a.pos, bd);
    const int* bt = resolve<const int>(a.bt, bd);
    const uint16_t* kv = resolve<const uint16_t>(a.kv, bd);
    const uint64_t pol = policy_evict_first();
    int i = 0;
    for (long long u = u0; ok && u < u1; ++u) {
      const int p = static_cast<int>(u / a.NB), blk = static_cast<int>(u % a.NB);
      const int r = p / a.Hkv, h = p % a.Hkv;
      const int ctxr = pos[r * a.T + a.T - 1] + 1;
      const int k0 = blk * kAttnKeys;
      if (k0 >= ctxr) continue;
      const int s = i % S;
      if (i >= S && !mbar_wait(&empty[s], ((i / S) - 1) & 1, ctx, 31)) {
        ok = false;
        break;
      }
      uint8_t* st = stage0 + s * L.stage_bytes;
      const int nk = min(kAttnKeys, ctxr - k0);
      if (a.P >= kAttnKeys) {
        const int lp = k0 / a.P;
        int page = lp < a.max_pages ? bt[static_cast<size_t>(r) * a.max_pages + lp] : -1;
        if (page < 0 || page >= a.num_pages) {
          report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 32, lp);
          page = 0;
        }
        const size_t kb = kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, h, k0 % a.P);
        const size_t vb = kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 1, h, k0 % a.P);
        mbar_arrive_expect_tx(&full[s], 2 * kAttnKeys * 256);
        bulk_load(st, kv + kb * 128, kAttnKeys * 256, &full[s], pol);
        bulk_load(st + kAttnKeys * 256, kv + vb * 128, kAttnKeys * 256, &full[s], pol);
      } else {
        const int npg = kAttnKeys / a.P;
        const int nvalid = min(npg, (nk + a.P - 1) / a.P);
        mbar_arrive_expect_tx(&full[s], 2 * nvalid * a.P * 256);
        for (int q = 0; q < nvalid; ++q) {
          const int lp = k0 / a.P + q;
          int page = lp < a.max_pages ? bt[static_cast<size_t>(r) * a.max_pages + lp] : -1;
          if (page < 0 || page >= a.num_pages) {
            report_error(ctx.status, DERR_BOUNDS, ctx.op_id, blockIdx.x, 33, lp);
            page = 0;
          }
          const size_t kb = kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 0, h, 0);
          const size_t vb = kv_row(a.layer, a.num_pages, a.Hkv, a.P, page, 1, h, 0);
          bulk_load(st + q * a.P * 256, kv + kb * 128, a.P * 256, &full[s], pol);
          bulk_load(st + kAttnKeys * 256 + q * a.P * 256, kv + vb * 128, a.P * 256, &full[s], pol);
        }
      }
      ++i;
    }
    const int issued = i;
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / S) * S;
      mbar_drain(&full[s], (last / S) & 1, ctx.budget_ns);
    }
    return;
  }

  // ---------------------------------------------------------- consumers
  const int ct = tid - 32, wc = warp - 1;  // wc: 0..7
  if (!group_wait(dep, ctx, 1, 256, ct == 0, 34, &flag[2])) return;
  const int* pos = resolve<const int>(a.pos, bd);
  const uint16_t* qg = static_cast<const uint16_t*>(a.q);
  const uint32_t qs_u32 = smem_u32(Qs), pb_u32 = smem_u32(Pb);
  const int tpr = 256 / QRp;             // softmax threads per row
  const int kpt = kAttnKeys / tpr;       // keys per softmax thread
  int i = 0;                             // valid-unit counter (matches producer)
  long long u = u0;
  while (u < u1) {
    const int p = static_cast<int>(u / a.NB);
    const int blk_a = static_cast<int>(u % a.NB);
    const long long run_end = min(u1, static_cast<long long>(p + 1) * a.NB);
    const int blk_b = static_cast<int>(run_end - static_cast<long long>(p) * a.NB);
    const int r = p / a.Hkv, h = p % a.Hkv;
    const int ctxr = pos[r * a.T + a.T - 1] + 1;
    // load this pair's query rows (swizzled 16-byte chunks) and positions
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
    for (int rr = ct; rr < QRp; rr += 256) {
      row_m[rr] = -INFINITY;
      row_l[rr] = 0.f;
      row_pos[rr] = rr < a.QR ? pos[r * a.T + rr / G] : -1;
    }
    float o[4][2][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    named_bar(1, 256);
    const int nvb = (ctxr + kAttnKeys - 1) / kAttnKeys;   // valid blocks
    for (int blk = blk_a; blk < min(blk_b, nvb); ++blk, ++i) {
      const int s = i % S;
      if (ct == 0) flag[2] = mbar_wait(&full[s], (i / S) & 1, ctx, 35) ? 1 : 0;
      named_bar(1, 256);
      if (!flag[2]) return;
      uint8_t* st = stage0 + s * L.stage_bytes;
      const uint32_t ks_u32 = smem_u32(st), vs_u32 = smem_u32(st + kAttnKeys * 256);
      const int k0 = blk * kAttnKeys;
      const int nk = min(kAttnKeys, ctxr - k0);
      if (nk < kAttnKeys) {
        // keys past the context were not loaded (or hold stale data): zero V
        for (int e = ct; e < (kAttnKeys - nk) * 16; e += 256)
          *reinterpret_cast<uint4*>(st + kAttnKeys * 256 + (nk + (e >> 4)) * 256 + (e & 15) * 16) =
              make_uint4(0, 0, 0, 0);
        fence_proxy_async_shared();  // ordered before the stage's next TMA fill
      }
      // S = Q K^T for keys [8 wc, 8 wc + 8) of the block
      {
        float sc[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[mt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
          uint32_t b0, b1, b2, b3;
          const int key = wc * 8 + (lane & 7);
          const int ch = ks * 2 + (lane >> 3);
          ldsm_x4(ks_u32 + key * 256 + ch * 16, b0, b1, b2, b3);
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            if (mt >= nmt) break;
            const int qrow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const int qch = (ks + kk) * 2 + (lane >> 4);
              uint32_t a0, a1, a2, a3;
              ldsm_x4(qs_u32 + qrow * 256 + ((qch ^ (qrow & 7)) << 4), a0, a1, a2, a3);
              if (kk == 0)
                mma_bf16_16816(sc[mt], a0, a1, a2, a3, b0, b1);
              else
                mma_bf16_16816(sc[mt], a0, a1, a2, a3, b2, b3);
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          if (mt >= nmt) break;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = mt * 16 + (lane >> 2) + (e >> 1) * 8;
            const int col = wc * 8 + (lane & 3) * 2 + (e & 1);
            const int key = k0 + col;
            const bool valid = rr < a.QR && key <= row_pos[rr] && col < nk;
            Sb[rr * kSPitch + col] = valid ? sc[mt][e] * a.scale_log2 : -INFINITY;
          }
        }
      }
      named_bar(1, 256);
      // online softmax: tpr threads per row
      {
        const int rr = ct / tpr, sub = ct % tpr;
        float sv[16];
        float lmax = -INFINITY;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (k >= kpt) break;
          sv[k] = Sb[rr * kSPitch + sub * kpt + k];
          lmax = fmaxf(lmax, sv[k]);
        }
        for (int o2 = tpr >> 1; o2 > 0; o2 >>= 1)
          lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o2));
        const float mold = row_m[rr];
        const float mnew = fmaxf(mold, lmax);
        const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(mold - mnew);
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          if (k >= kpt) break;
          const float pv = (mnew == -INFINITY) ? 0.f : exp2f(sv[k] - mnew);
          lsum += pv;
          const int col = sub * kpt + k;
          const int ch = col >> 3;
          Pb[(rr * 128 + (((ch ^ (rr & 7)) << 4) + (col & 7) * 2)) >> 1] = f2bf(pv);
        }
        for (int o2 = tpr >> 1; o2 > 0; o2 >>= 1)
          lsum += __shfl_xor_sync(0xffffffffu, lsum, o2);
        named_bar(1, 256);   // everyone has read row_m before it changes
        if (sub == 0) {
          row_sc[rr] = alpha;
          row_m[rr] = mnew;
          row_l[rr] = row_l[rr] * alpha + lsum;
        }
      }
      named_bar(1, 256);
      // O = O * alpha + P V for d columns [16 wc, 16 wc + 16)
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        if (mt >= nmt) break;
        const float s0 = row_sc[mt * 16 + (lane >> 2)];
        const float s1 = row_sc[mt * 16 + (lane >> 2) + 8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          o[mt][nt][0] *= s0;
          o[mt][nt][1] *= s0;
          o[mt][nt][2] *= s1;
          o[mt][nt][3] *= s1;
        }
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t b0, b1, b2, b3;
        const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = wc * 2 + (lane >> 4);
        ldsm_x4_t(vs_u32 + key * 256 + ch * 16, b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          if (mt >= nmt) break;
          const int prow = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int pch = ks * 2 + (lane >> 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(pb_u32 + prow * 128 + ((pch ^ (prow & 7)) << 4), a0, a1, a2, a3);
          mma_bf16_16816(o[mt][0], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o[mt][1], a0, a1, a2, a3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // ---- finish this pair: normalised partial O and its lse (base 2)
    named_bar(1, 256);
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      if (mt >= nmt) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = mt * 16 + (lane >> 2) + (e >> 1) * 8;
        const float l = row_l[rr];
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          Ob[rr * 128 + wc * 16 + nt * 8 + (lane & 3) * 2 + (e & 1)] = o[mt][nt][e] * inv;
      }
    }
    for (int rr = ct; rr < QRp; rr += 256) {
      const float l = row_l[rr];
      row_lse[rr] = l > 0.f ? row_m[rr] + log2f(l) : -INFINITY;
    }
    named_bar(1, 256);
    const bool whole = (blk_a == 0 && blk_b == a.NB);
    if (!whole) {
      const long long ps = static_cast<long long>(p) * a.NB;
      const int slot = (u >= ps) ? 0 : 1;
      const size_t part = static_cast<size_t>(QRp) * 129;
      float* mine = a.ws + static_cast<size_t>(c * 2 + slot) * part;
      for (int e = ct; e < QRp * 128; e += 256) mine[e] = Ob[e];
      for (int rr = ct; rr < QRp; rr += 256) mine[QRp * 128 + rr] = row_lse[rr];
      __threadfence();
      named_bar(1, 256);
      const int cf = sk_owner(U, a.G, ps), cl = sk_owner(U, a.G, ps + a.NB - 1);
      if (ct == 0) {
        int n = 0;
        for (int cc = cf; cc <= cl; ++cc)
          if (sk_begin(U, a.G, cc + 1) > sk_begin(U, a.G, cc)) ++n;
        const unsigned old = atomicAdd(a.pair_cnt + p, 1u);
        flag[0] = (old + 1 == static_cast<unsigned>(n)) ? 1 : 0;
      }
      named_bar(1, 256);
      if (flag[0]) {
        __threadfence();
        // per-row weights of every contributor: w_i = 2^(lse_i - max)
        for (int rr = ct; rr < QRp; rr += 256) {
          float mx = -INFINITY;
          for (int cc = cf; cc <= cl; ++cc) {
            const long long b0 = sk_begin(U, a.G, cc);
            if (sk_begin(U, a.G, cc + 1) <= b0) continue;
            const int sl = (b0 >= ps) ? 0 : 1;
            const float le = cc == c ? row_lse[rr]
                                     : __ldcg(a.ws + static_cast<size_t>(cc * 2 + sl) * part + QRp * 128 + rr);
            mx = fmaxf(mx, le);
          }
          row_w[rr] = mx;
        }
        named_bar(1, 256);
        for (int e = ct; e < QRp * 128; e += 256) {
          const int rr = e >> 7;
          const float mx = row_w[rr];
          float num = 0.f, den = 0.f;
          if (mx != -INFINITY) {
            for (int cc = cf; cc <= cl; ++cc) {
              const long long b0 = sk_begin(U, a.G, cc);
              if (sk_begin(U, a.G, cc + 1) <= b0) continue;
              const int sl = (b0 >= ps) ? 0 : 1;
              const float* src = a.ws + static_cast<size_t>(cc * 2 + sl) * part;
              const float le = cc == c ? row_lse[rr] : __ldcg(src + QRp * 128 + rr);
              const float ov = cc == c ? Ob[e] : __ldcg(src + e);
              const float wgt = exp2f(le - mx);
              num = fmaf(wgt, ov, num);
              den += wgt;
            }
          }
          Ob[e] = den > 0.f ? num / den : 0.f;
        }
        if (ct == 0) a.pair_cnt[p] = 0u;
        named_bar(1, 256);
      }
    }
    if (whole || flag[0]) {
      // write the attention output, one warp per query row
      for (int rr = wc; rr < a.QR; rr += 8) {
        const int t = rr / G, g = rr % G;
        const size_t m = static_cast<size_t>(r) * a.T + t;
        const int hq = h * G + g;
        const float4 v = *reinterpret_cast<const float4*>(Ob + rr * 128 + lane * 4);
        if (!a.fp8) {
          uint16_t* out = static_cast<uint16_t*>(a.out) + (m * a.Hq + hq) * 128 + lane * 4;
          const uint32_t lo = static_cast<uint32_t>(f2bf(v.x)) | (static_cast<uint32_t>(f2bf(v.y)) << 16);
          const uint32_t hi = static_cast<uint32_t>(f2bf(v.z)) | (static_cast<uint32_t>(f2bf(v.w)) << 16);
          *reinterpret_cast<uint2*>(out) = make_uint2(lo, hi);
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
    }
    named_bar(1, 256);
    u = run_end;
  }
}

}  // namespace dl
