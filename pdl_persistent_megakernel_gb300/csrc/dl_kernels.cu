// dl_kernels.cu -- the kernels: one standalone kernel per operation family
// (serial and graph schedules) and the persistent tile-instruction
// megakernel.  All of them run the tile engines of dl_ops.cuh.
#include <cuda_runtime.h>

#include "dl_kernels.h"
#include "dl_ops.cuh"

namespace dl {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t*>((a + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ int tmem_cols_pow2(int cols) {
  int n = 32;
  while (n < cols) n <<= 1;
  return n;
}

// ------------------------------------------------------------ standalone
// kS > 1: launched in clusters of kS CTAs, one row per cluster
template <int NV, int kS>
__global__ void __launch_bounds__(kThreads, 1) k_norm(NormArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  Dep dep{};
  dep.mode = 0;
  norm_op<NV, true, kS>(a, blockIdx.x, dep, ctx, align1024(smem_raw));
}

template <int kMG, int kMp>
__global__ void __launch_bounds__(kThreads, 1) k_gemm(GemmArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  if (a.gdc_mode == 2) gdc_wait();   // ablation: wait at entry, before the prologue
  uint8_t* smem = align1024(smem_raw);
  uint32_t tmem = 0;
  int cols = 0;
  if constexpr (kMp > 0) {
    cols = tmem_cols_pow2(a.tmem_bufs * (a.pair ? 2 : 1) * kMp);
    if ((threadIdx.x >> 5) == 1) {
      tmem_alloc(&tmem_slot, cols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    tmem = tmem_slot;
  }
  Dep dep{};
  dep.mode = 0;
  gemm_op_t<kMG, kMp>(a, blockIdx.x, dep, ctx, smem, tmem);
  if constexpr (kMp > 0) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) tmem_dealloc(tmem, cols);
  }
}

template <int kNMT>
__global__ void __launch_bounds__(kThreads, 1) k_attn(AttnArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  Dep dep{};
  dep.mode = 0;
  attn_op_t<kNMT, false>(a, blockIdx.x, dep, ctx, align1024(smem_raw), 0u);
}

// tcgen05 attention: 512 TMEM columns (two O, two S buffers) for the CTA.
__global__ void __launch_bounds__(kThreads, 1) k_attn_tc(AttnArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  Dep dep{};
  dep.mode = 0;
  attn_op_t<1, true>(a, blockIdx.x, dep, ctx, align1024(smem_raw), tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 1) tmem_dealloc(tmem, 512);
}

__global__ void k_bind(Binding* dst, Binding v) { *dst = v; }

// Test-only pure copies through the paged-cache slot math (bit-exact).
__global__ void k_test_kv_write(const uint16_t* src, uint16_t* kv, const int* bt,
                                const int* pos, int layer, int M, int T, int Hkv,
                                int d, int P, int num_pages, int max_pages,
                                DevStatus* st) {
  const int m = blockIdx.x / (2 * Hkv), kvsel = (blockIdx.x / Hkv) % 2, h = blockIdx.x % Hkv;
  if (m >= M) return;
  const int p = pos[m], r = m / T, lp = p / P;
  const int page = (lp >= 0 && lp < max_pages) ? bt[static_cast<size_t>(r) * max_pages + lp] : -1;
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) report_error(st, DERR_BOUNDS, 0, blockIdx.x, 50, lp);
    return;
  }
  const size_t dst = kv_row(layer, num_pages, Hkv, P, page, kvsel, h, p % P) * d;
  const size_t s0 = ((static_cast<size_t>(m) * 2 + kvsel) * Hkv + h) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) kv[dst + i] = src[s0 + i];
}

__global__ void k_test_kv_gather(const uint16_t* kv, const int* bt, uint16_t* dst,
                                 int layer, int R, int n_keys, int Hkv, int d, int P,
                                 int num_pages, int max_pages, DevStatus* st) {
  const long long row = blockIdx.x;  // (r, kv, h, j)
  const int j = static_cast<int>(row % n_keys);
  const int h = static_cast<int>((row / n_keys) % Hkv);
  const int kvsel = static_cast<int>((row / (static_cast<long long>(n_keys) * Hkv)) % 2);
  const int r = static_cast<int>(row / (2LL * n_keys * Hkv));
  if (r >= R) return;
  const int lp = j / P;
  const int page = lp < max_pages ? bt[static_cast<size_t>(r) * max_pages + lp] : -1;
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) report_error(st, DERR_BOUNDS, 0, blockIdx.x, 51, lp);
    return;
  }
  const size_t src = kv_row(layer, num_pages, Hkv, P, page, kvsel, h, j % P) * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) dst[row * d + i] = kv[src + i];
}

// ------------------------------------------------------------ megakernel
// One worker CTA per SM walks its host-built queue.  Warp 0 is the producer:
// it runs ahead of the other warps across instruction boundaries and fills
// the worker's ring of operand slots in the order they will be consumed
// (weights at once, dependent data once the instruction's event counters
// are reached).  Warps 1-8 consume instruction after instruction: before
// an instruction's dependent reads they acquire-poll the event counters it
// names; after it, one thread publishes with a release add.  Instructions
// only wait on earlier instructions of a global topological order and all
// workers are co-resident (cooperative launch), so the earliest unfinished
// instruction can always run; the producer never blocks on a slot that only
// the consumption of its own pending (dependent) loads could free.
__global__ void __launch_bounds__(kThreads, 1) k_mega(MegaArgs m, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(16) Instr ins;
  __shared__ __align__(16) OpArgs op;
  __shared__ int stop;
  __shared__ __align__(8) uint64_t ring_full[kMaxSlots], ring_empty[kMaxSlots];
  __shared__ __align__(8) uint64_t tbars[12];   // TMEM full[4], empty[4]; tile ready[2], free[2]
  __shared__ int p_pgbuf[32 * 4], p_ppos[kMaxM];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* priv = smem + m.priv_off;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int kTmemCols = 512;   // one worker per SM owns all of TMEM
  if (tid == 0) {
    for (int s = 0; s < m.ns; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 8);
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(&tbars[b], 1);
      mbar_init(&tbars[4 + b], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tbars[8 + b], 4);
      mbar_init(&tbars[10 + b], 2);
    }
    stop = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  Pipe R;
  R.base = smem;
  R.full = ring_full;
  R.empty = ring_empty;
  R.slot_bytes = static_cast<uint32_t>(m.slot_bytes);
  pipe_set_ns(R, static_cast<uint32_t>(m.ns));
  R.seq0 = 0;
  R.ups = 1;
  R.x_bytes = 0;
  R.empty_cnt = 8;
  const Instr* q = m.queues + static_cast<size_t>(blockIdx.x) * m.qlen;

  if (warp == 0) {
    // --------------------------------------------------------- producer
    uint32_t seq = 0, hi = 0;
    bool ok = true;
    for (int pc = 0; pc < m.qlen && ok; ++pc) {
      const Instr* in = q + pc;
      const uint32_t row = __ldg(&in->op_row);
      if (row == 0xffffffffu) break;
      const OpArgs* oa = m.ops + row;
      const int kind = __ldg(&oa->kind);
      Dep dep{};
      dep.mode = 1;
      dep.n = static_cast<int>(__ldg(&in->n_wait));
      for (int i = 0; i < dep.n && i < 4; ++i) {
        dep.ev[i] = m.events + __ldg(&in->wait_event[i]);
        dep.val[i] = __ldg(&in->wait_value[i]);
      }
      KernelCtx c2 = ctx;
      c2.op_id = static_cast<int>(row);
      const int cta = static_cast<int>(__ldg(&in->cta));
      if (kind == OP_GEMM) {
        const GemmArgs& ga = oa->gemm;
        if (lane == 0) ok = mk_produce_gemm(ga, cta, dep, c2, R, seq, &hi);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        const int ups = ga.pair ? 1 : 2;
        seq += static_cast<uint32_t>((gemm_share_units(ga, cta) + ups - 1) / ups);
      } else if (kind == OP_ATTN) {
        int nv = 0;
        ok = mk_produce_attn(oa->attn, cta, dep, c2, R, seq, p_pgbuf, p_ppos, &nv, &hi);
        seq += static_cast<uint32_t>(nv);
      }
      if (aborted(ctx.status)) ok = false;
      __syncwarp();
    }
    // no copy may be in flight when the worker leaves
    if (lane == 0) {
      const uint32_t lo = hi > R.ns ? hi - R.ns : 0u;
      for (uint32_t s = lo; s < hi; ++s)
        mbar_drain(pipe_full(R, s), pipe_par(R, s), ctx.budget_ns);
    }
  } else {
    // ------------------------------------------------------- consumers
    const int ct = tid - 32;
    uint32_t seq = 0, tseq = 0, rseq = 0;
    for (int pc = 0; pc < m.qlen; ++pc) {
      if (ct < 32) reinterpret_cast<uint32_t*>(&ins)[ct] = __ldg(reinterpret_cast<const uint32_t*>(q + pc) + ct);
      named_bar(1, 256);
      if (ins.op_row == 0xffffffffu) break;   // NoOp padding: the queue is done
      for (int i = ct; i < static_cast<int>(sizeof(OpArgs) / 4); i += 256)
        reinterpret_cast<uint32_t*>(&op)[i] = __ldg(reinterpret_cast<const uint32_t*>(m.ops + ins.op_row) + i);
      named_bar(1, 256);
      Dep dep{};
      dep.mode = 1;
      dep.n = static_cast<int>(ins.n_wait);
      for (int i = 0; i < dep.n && i < 4; ++i) {
        dep.ev[i] = m.events + ins.wait_event[i];
        dep.val[i] = ins.wait_value[i];
      }
      KernelCtx c2 = ctx;
      c2.op_id = static_cast<int>(ins.op_row);
      const int cta = static_cast<int>(ins.cta);
      if (m.trace && ct == 0)
        m.trace[(static_cast<size_t>(blockIdx.x) * m.qlen + pc) * 4 + 0] =
            static_cast<unsigned>(globaltimer());
      bool fail = false;
      switch (op.kind) {
        case OP_NORM:
          mk_norm(op.norm, cta, dep, c2, priv);
          break;
        case OP_GEMM: {
          const int ups = op.gemm.pair ? 1 : 2;
          Pipe P = R;
          P.seq0 = seq;
          P.ups = ups;
          P.x_bytes = ((op.gemm.Mp * 128 + 1023) / 1024) * 1024;
          TmemRing TR;
          TR.base = tmem;
          TR.nbuf = 4;
          TR.nbuf_magic = fdiv_magic(4u);
          TR.stride = 128;
          TR.seq0 = tseq;
          TR.rseq0 = rseq;
          mk_gemm(op.gemm, cta, dep, c2, priv, P, TR, tbars);
          const int n = gemm_share_units(op.gemm, cta);
          seq += static_cast<uint32_t>((n + ups - 1) / ups);
          if (op.gemm.mma) {
            tseq += static_cast<uint32_t>(n);
            rseq += static_cast<uint32_t>(gemm_share_handoffs(op.gemm, cta));
          }
          break;
        }
        case OP_ATTN: {
          Pipe P = R;
          P.seq0 = seq;
          P.ups = 1;
          const int nv = mk_attn(op.attn, cta, dep, c2, priv, P);
          if (nv < 0)
            fail = true;
          else
            seq += static_cast<uint32_t>(nv);
          break;
        }
        default:
          if (ct == 0) report_error(ctx.status, DERR_BAD_OP, ins.op_row, blockIdx.x, 40, op.kind);
          break;
      }
      named_bar(1, 256);
      if (ct == 0) {
        const bool ab = fail || aborted(ctx.status);
        if (!ab) {
          fence_proxy_async_global();
          __threadfence();
          for (uint32_t s = 0; s < ins.n_signal && s < kMaxSignals; ++s)
            red_release_gpu_add(m.events + instr_signal_event(ins, s), instr_signal_inc(ins, s));
        }
        stop = ab ? 1 : 0;
        if (m.trace)
          m.trace[(static_cast<size_t>(blockIdx.x) * m.qlen + pc) * 4 + 2] =
              static_cast<unsigned>(globaltimer());
      }
      named_bar(1, 256);
      if (stop) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // the last worker out zeroes the event counters for the next step
  if (tid == 0) {
    __threadfence();
    const unsigned old = atomicAdd(m.finish_cnt, 1u);
    if (old + 1 == gridDim.x) {
      for (int e = 0; e < m.num_events; ++e) m.events[e] = 0u;
      *m.finish_cnt = 0u;
      __threadfence();
    }
  }
}

// ------------------------------------------------------------ host side
const void* gemm_kernel(int mma, int m_or_mp) {
  if (!mma) {
    if (m_or_mp <= 1) return reinterpret_cast<const void*>(&k_gemm<1, 0>);
    if (m_or_mp <= 2) return reinterpret_cast<const void*>(&k_gemm<2, 0>);
    return reinterpret_cast<const void*>(&k_gemm<4, 0>);
  }
  if (m_or_mp <= 16) return reinterpret_cast<const void*>(&k_gemm<0, 16>);
  if (m_or_mp <= 32) return reinterpret_cast<const void*>(&k_gemm<0, 32>);
  return reinterpret_cast<const void*>(&k_gemm<0, 64>);
}

const void* norm_kernel(int H, int split) {
  const int nv = ((H >> 3) / split + 255) >> 8;
  if (split == 4) return nv <= 1 ? reinterpret_cast<const void*>(&k_norm<1, 4>) : nullptr;
  if (split == 2) return nv <= 1 ? reinterpret_cast<const void*>(&k_norm<1, 2>) : nullptr;
  if (split != 1) return nullptr;
  if (nv <= 1) return reinterpret_cast<const void*>(&k_norm<1, 1>);
  if (nv <= 2) return reinterpret_cast<const void*>(&k_norm<2, 1>);
  return reinterpret_cast<const void*>(&k_norm<4, 1>);
}
const void* attn_tc_kernel() { return reinterpret_cast<const void*>(&k_attn_tc); }

int attn_tc_smem_bytes(int QRp, int stages) {
  return attn_tc_smem_layout(QRp, stages).total + 1024;
}

const void* attn_kernel(int QRp) {
  if (QRp <= 16) return reinterpret_cast<const void*>(&k_attn<1>);
  if (QRp <= 32) return reinterpret_cast<const void*>(&k_attn<2>);
  return reinterpret_cast<const void*>(&k_attn<4>);
}
const void* mega_kernel() { return reinterpret_cast<const void*>(&k_mega); }

cudaError_t launch_bind(Binding* dst, const Binding& v, cudaStream_t s) {
  k_bind<<<1, 1, 0, s>>>(dst, v);
  return cudaGetLastError();
}

int gemm_smem_bytes(int npair, int Mp, int stages, int KB, int fp8, int epi, int M, int share) {
  return gemm_smem_layout(npair, Mp, stages, KB, fp8, epi, M, share).total + 1024;
}

int attn_smem_bytes(int QRp, int stages) {
  return attn_smem_layout(QRp, stages).total + 1024;
}

// the reduction scratch, the contributor table of a deferred fix-up (up to
// 64 tiles of 128 columns) and the norm weight (H <= 8192 bf16)
int norm_smem_bytes() { return 1024 + kNormWOff + 8192 * 2; }

cudaError_t launch_test_kv_write(const void* src, void* kv, const int* bt, const int* pos,
                                 int layer, int M, int T, int Hkv, int d, int P,
                                 int num_pages, int max_pages, DevStatus* st,
                                 cudaStream_t s) {
  k_test_kv_write<<<M * 2 * Hkv, 128, 0, s>>>(static_cast<const uint16_t*>(src),
                                              static_cast<uint16_t*>(kv), bt, pos, layer, M, T,
                                              Hkv, d, P, num_pages, max_pages, st);
  return cudaGetLastError();
}

cudaError_t launch_test_kv_gather(const void* kv, const int* bt, void* dst, int layer, int R,
                                  int n_keys, int Hkv, int d, int P, int num_pages,
                                  int max_pages, DevStatus* st, cudaStream_t s) {
  const long long rows = 2LL * R * Hkv * n_keys;
  k_test_kv_gather<<<static_cast<unsigned>(rows), 128, 0, s>>>(
      static_cast<const uint16_t*>(kv), bt, static_cast<uint16_t*>(dst), layer, R, n_keys, Hkv,
      d, P, num_pages, max_pages, st);
  return cudaGetLastError();
}

}  // namespace dl
