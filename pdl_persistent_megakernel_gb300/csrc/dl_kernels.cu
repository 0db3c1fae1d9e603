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
__global__ void __launch_bounds__(kThreads, 1) k_norm(NormArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  Dep dep{};
  dep.mode = 0;
  norm_op(a, blockIdx.x, dep, ctx, align1024(smem_raw));
}

template <int kMG, int kMp>
__global__ void __launch_bounds__(kThreads, 1) k_gemm(GemmArgs a, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
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
  attn_op_t<kNMT>(a, blockIdx.x, dep, ctx, align1024(smem_raw));
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
// Runs one GEMM instruction with the variant its arguments call for.
__device__ void mega_gemm(const GemmArgs& a, int c, const Dep& dep,
                          const KernelCtx& ctx, uint8_t* smem, uint32_t tmem) {
  if (!a.mma) {
    if (a.M <= 1)
      gemm_op_t<1, 0>(a, c, dep, ctx, smem, tmem);
    else if (a.M <= 2)
      gemm_op_t<2, 0>(a, c, dep, ctx, smem, tmem);
    else
      gemm_op_t<4, 0>(a, c, dep, ctx, smem, tmem);
  } else {
    if (a.Mp <= 16)
      gemm_op_t<0, 16>(a, c, dep, ctx, smem, tmem);
    else if (a.Mp <= 32)
      gemm_op_t<0, 32>(a, c, dep, ctx, smem, tmem);
    else
      gemm_op_t<0, 64>(a, c, dep, ctx, smem, tmem);
  }
}

// One worker CTA per SM walks its host-built queue.  Before an instruction's
// dependent reads it acquire-polls the event counters the instruction names
// (weights are prefetched first); after it, thread 0 publishes with a
// release add.  Instructions only wait on earlier instructions of a global
// topological order and all workers are co-resident (cooperative launch), so
// the earliest unfinished instruction can always run.
__global__ void __launch_bounds__(kThreads, 1) k_mega(MegaArgs m, KernelCtx ctx) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(16) Instr ins;
  __shared__ __align__(16) OpArgs op;
  __shared__ int stop;
  uint8_t* smem = align1024(smem_raw);
  const int tid = threadIdx.x;
  constexpr int kTmemCols = 512;   // one worker per SM owns all of TMEM
  if ((tid >> 5) == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const Instr* q = m.queues + static_cast<size_t>(blockIdx.x) * m.qlen;
  for (int pc = 0; pc < m.qlen; ++pc) {
    if (tid < 32) reinterpret_cast<uint32_t*>(&ins)[tid] = __ldg(reinterpret_cast<const uint32_t*>(q + pc) + tid);
    __syncthreads();
    if (ins.op_row == 0xffffffffu) break;   // NoOp padding: the queue is done
    for (int i = tid; i < static_cast<int>(sizeof(OpArgs) / 4); i += kThreads)
      reinterpret_cast<uint32_t*>(&op)[i] = __ldg(reinterpret_cast<const uint32_t*>(m.ops + ins.op_row) + i);
    __syncthreads();
    Dep dep{};
    dep.mode = 1;
    dep.n = static_cast<int>(ins.n_wait);
    for (int i = 0; i < dep.n && i < 4; ++i) {
      dep.ev[i] = m.events + ins.wait_event[i];
      dep.val[i] = ins.wait_value[i];
    }
    KernelCtx c2 = ctx;
    c2.op_id = static_cast<int>(ins.op_row);
    if (m.trace && tid == 0)
      m.trace[(static_cast<size_t>(blockIdx.x) * m.qlen + pc) * 4 + 0] =
          static_cast<unsigned>(globaltimer());
    switch (op.kind) {
      case OP_NORM:
        norm_op(op.norm, static_cast<int>(ins.cta), dep, c2, smem);
        break;
      case OP_GEMM:
        mega_gemm(op.gemm, static_cast<int>(ins.cta), dep, c2, smem, tmem);
        break;
      case OP_ATTN:
        attn_op(op.attn, static_cast<int>(ins.cta), dep, c2, smem);
        break;
      default:
        if (tid == 0) report_error(ctx.status, DERR_BAD_OP, ins.op_row, blockIdx.x, 40, op.kind);
        break;
    }
    __syncthreads();
    if (tid == 0) {
      const bool ab = aborted(ctx.status);
      if (!ab) {
        fence_proxy_async_global();
        __threadfence();
        for (uint32_t s = 0; s < ins.n_signal && s < 2; ++s)
          red_release_gpu_add(m.events + ins.signal_event[s], ins.signal_inc[s]);
      }
      stop = ab ? 1 : 0;
      if (m.trace)
        m.trace[(static_cast<size_t>(blockIdx.x) * m.qlen + pc) * 4 + 2] =
            static_cast<unsigned>(globaltimer());
    }
    __syncthreads();
    if (stop) break;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((tid >> 5) == 1) tmem_dealloc(tmem, kTmemCols);
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

const void* norm_kernel() { return reinterpret_cast<const void*>(&k_norm); }
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

int gemm_smem_bytes(int npair, int Mp, int stages, int KB, int fp8, int epi, int M) {
  return gemm_smem_layout(npair, Mp, stages, KB, fp8, epi, M).total + 1024;
}

int attn_smem_bytes(int QRp, int stages) {
  return attn_smem_layout(QRp, stages).total + 1024;
}

int norm_smem_bytes() { return 1024 + 256; }

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
