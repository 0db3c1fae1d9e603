// dl_bench.cu -- microbenchmarks of the mechanisms the schedules are built
// from, measured in isolation on the device:
//   - the cost of one tcgen05.mma at the decode step's shapes (M = 128,
//     N = 16..256, bf16 K = 16 or e4m3 K = 32 per instruction), issued into
//     one or several TMEM accumulators by one or two threads;
//   - the round trip of a release-add / acquire-poll hand-off between two
//     CTAs on different SMs (the megakernel's event protocol, page
//     "Kernel-Mega-PDL", section 4: gmem counters published with release
//     atomics and awaited with acquire polling).
// Every wait is bounded by a %globaltimer budget and reported, never spun on
// forever; the TMEM the MMA kernel allocates is released before it returns.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "dl.h"
#include "dl_device.cuh"
#include "dl_internal.h"

namespace dl {
dl_status set_last_error(dl_status s, const char* msg);  // dl_host.cu
}

using namespace dl;

namespace {

constexpr unsigned long long kBenchBudgetNs = 200000000ull;   // 0.2 s per wait

// out[0] = ns from the first MMA's issue to the completion of the last,
// out[1] = 1 if a wait gave up.  One CTA of 128 threads; the operands are
// zero tiles in shared memory (A: 128 rows x 128 B, B: n rows x 128 B, both
// K-major with the 128-byte swizzle).
__global__ void __launch_bounds__(128, 1) k_bench_mma(int fp8, int n, int n_mma, int n_acc,
                                                      int n_issuers, int lean,
                                                      unsigned long long* out) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t done[2];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  // zero A (16 KiB) and B (n x 128 B)
  const int bytes = 16384 + n * 128;
  for (int e = tid * 16; e < bytes; e += 128 * 16)
    *reinterpret_cast<uint4*>(smem + e) = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    mbar_init(&done[0], 1);
    mbar_init(&done[1], 1);
    fence_barrier_init();
  }
  fence_proxy_async_shared();
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t sa = smem_u32(smem), sb = smem_u32(smem + 16384);
  const uint32_t idesc = umma_idesc(n, fp8 == 0);
  bool ok = true;
  unsigned long long t0 = 0, t1 = 0;
  const int w = warp;   // issuer index: lane 0 of warps 0 .. n_issuers - 1
  if (w < n_issuers && (tid & 31) == 0 && lean) {
    // lean issue: descriptors built once and advanced by constants (the
    // start-address field counts 16-byte units: +32 bytes = +2), four MMAs
    // per pass into this issuer's accumulator, nothing else in the loop
    const uint64_t ad0 = umma_desc_sw128(sa), bd0 = umma_desc_sw128(sb);
    const uint32_t d = tmem + static_cast<uint32_t>((w % n_acc) * n);
    t0 = globaltimer();
    for (int i = w * 4; i < n_mma; i += n_issuers * 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (fp8)
          umma_e4m3(d, ad0 + 2 * k, bd0 + 2 * k, idesc, (i + k) > 0 ? 1u : 0u);
        else
          umma_bf16(d, ad0 + 2 * k, bd0 + 2 * k, idesc, (i + k) > 0 ? 1u : 0u);
      }
    }
    umma_commit(&done[w]);
    const unsigned long long ts = globaltimer();
    while (!mbar_try_wait(&done[w], 0)) {
      if (globaltimer() - ts > kBenchBudgetNs) {
        ok = false;
        break;
      }
    }
    t1 = globaltimer();
  } else if (w < n_issuers && (tid & 31) == 0) {
    t0 = globaltimer();
    int k = 0;
    for (int i = w; i < n_mma; i += n_issuers, ++k) {
      const int acc = i % n_acc;
      const uint32_t d = tmem + static_cast<uint32_t>(acc * n);
      const uint64_t ad = umma_desc_sw128(sa + (k & 3) * 32);
      const uint64_t bd = umma_desc_sw128(sb + (k & 3) * 32);
      const uint32_t accumulate = i >= n_acc ? 1u : 0u;
      if (fp8)
        umma_e4m3(d, ad, bd, idesc, accumulate);
      else
        umma_bf16(d, ad, bd, idesc, accumulate);
    }
    umma_commit(&done[w]);
    const unsigned long long ts = globaltimer();
    while (!mbar_try_wait(&done[w], 0)) {
      if (globaltimer() - ts > kBenchBudgetNs) {
        ok = false;
        break;
      }
    }
    t1 = globaltimer();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
  if (tid == 0 || (tid == 32 && n_issuers > 1)) {
    // the slower issuer's span (both start together after the barrier)
    atomicMax(&out[0], t1 - t0);
    if (!ok) atomicExch(&out[1], 1ull);
  }
}

// Two CTAs (a cooperative launch, so both are resident) hand a token back
// and forth through one global counter: CTA 0 adds 1 (release) and polls
// (acquire) for the reply, CTA 1 polls for the token and adds 1.
// out[0] = ns for `iters` round trips, out[1] = 1 if a poll gave up.
__global__ void k_bench_poll(unsigned* flag, int iters, unsigned long long* out) {
  if (threadIdx.x != 0) return;
  const bool ping = blockIdx.x == 0;
  bool ok = true;
  const unsigned long long t0 = globaltimer();
  for (int i = 0; i < iters && ok; ++i) {
    const unsigned want = ping ? 2u * i + 2u : 2u * i + 1u;
    if (ping) red_release_gpu_add(flag, 1u);
    const unsigned long long ts = globaltimer();
    while (ld_acquire_gpu(flag) < want) {
      if (globaltimer() - ts > kBenchBudgetNs) {
        ok = false;
        break;
      }
    }
    if (!ping && ok) red_release_gpu_add(flag, 1u);
  }
  const unsigned long long t1 = globaltimer();
  if (ping) out[0] = t1 - t0;
  if (!ok) atomicExch(&out[1], 1ull);
}

dl_status bench_err(dl_status s, const char* what, cudaError_t e = cudaSuccess) {
  char buf[200];
  std::snprintf(buf, sizeof(buf), "%s%s%s", what, e != cudaSuccess ? ": " : "",
                e != cudaSuccess ? cudaGetErrorString(e) : "");
  return set_last_error(s, buf);
}

}  // namespace

extern "C" dl_status dl_bench_mma(int fp8, int n, int n_mma, int n_accumulators, int n_issuers,
                                  int lean, double* ns_per_mma) {
  if (!ns_per_mma) return bench_err(DL_ERR_INVALID_ARG, "dl_bench_mma: NULL output");
  if (n < 16 || n > 256 || n % 16 || n_mma < 4 || n_mma > 65536 || n_mma % 4 || n_accumulators < 1 ||
      n_accumulators * n > 512 || n_issuers < 1 || n_issuers > 2)
    return bench_err(DL_ERR_INVALID_ARG,
                     "dl_bench_mma: n in 16..256 (multiple of 16), n_accumulators * n <= 512, "
                     "1 or 2 issuers, n_mma a multiple of 4 in 4..65536");
  unsigned long long* d_out = nullptr;
  cudaError_t e = cudaMalloc(&d_out, 2 * sizeof(unsigned long long));
  if (e != cudaSuccess) return bench_err(DL_ERR_OOM, "dl_bench_mma: cudaMalloc", e);
  unsigned long long h[2] = {0, 0};
  const int smem = 1024 + 16384 + 256 * 128;
  e = cudaFuncSetAttribute(k_bench_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaMemset(d_out, 0, sizeof(h));
  if (e == cudaSuccess) {
    k_bench_mma<<<1, 128, smem>>>(fp8 ? 1 : 0, n, n_mma, n_accumulators, n_issuers,
                                  lean ? 1 : 0, d_out);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d_out);
  if (e != cudaSuccess) return bench_err(DL_ERR_CUDA, "dl_bench_mma", e);
  if (h[1]) return bench_err(DL_ERR_TIMEOUT, "dl_bench_mma: the MMA completion wait gave up");
  *ns_per_mma = static_cast<double>(h[0]) / n_mma;
  return DL_OK;
}

extern "C" dl_status dl_bench_poll_latency(int iters, double* ns_per_round_trip) {
  if (!ns_per_round_trip || iters < 1 || iters > (1 << 20))
    return bench_err(DL_ERR_INVALID_ARG, "dl_bench_poll_latency: 1 <= iters <= 2^20, output");
  int dev = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return bench_err(DL_ERR_CUDA, "dl_bench_poll_latency", e);
  if (!coop) return bench_err(DL_ERR_UNSUPPORTED, "dl_bench_poll_latency: no cooperative launch");
  unsigned* d_flag = nullptr;
  unsigned long long* d_out = nullptr;
  e = cudaMalloc(&d_flag, 256);
  if (e == cudaSuccess) e = cudaMalloc(&d_out, 2 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(d_flag, 0, 256);
  if (e == cudaSuccess) e = cudaMemset(d_out, 0, 2 * sizeof(unsigned long long));
  unsigned long long h[2] = {0, 0};
  if (e == cudaSuccess) {
    void* args[] = {&d_flag, &iters, &d_out};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_bench_poll), dim3(2),
                                    dim3(32), args, 0, nullptr);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d_flag);
  cudaFree(d_out);
  if (e != cudaSuccess) return bench_err(DL_ERR_CUDA, "dl_bench_poll_latency", e);
  if (h[1]) return bench_err(DL_ERR_TIMEOUT, "dl_bench_poll_latency: a poll gave up");
  *ns_per_round_trip = static_cast<double>(h[0]) / iters;
  return DL_OK;
}
