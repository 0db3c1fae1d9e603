// dl_noalloc.cu -- split-KV attention of one layer through a fixed,
// statically reserved scratch area instead of plan-owned device memory.
//
// Some callers cannot allocate device memory at the point where they want
// the attention: a framework that owns the device allocator and forbids
// foreign cudaMalloc calls, a caller whose memory-pool budget is already
// spent, or one that must not pay the implicit synchronisation cudaFree
// brings.  For them this entry point takes everything it needs (the
// binding table with the cache's TMA descriptor, the device status word,
// the per-(request, kv head) arrival counters and the fp32 split-KV
// partials) from one file-scope __device__ array whose size is fixed at
// build time.  It launches the split-KV attention kernel on the mma.sync
// engine (the one the megakernel runs, and the standalone schedules under
// DL_ATTN=mma_sync) with the plans' work split and pipeline depth; only the
// origin of its scratch differs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "dl.h"
#include "dl_internal.h"
#include "dl_kernels.h"

namespace dl {
dl_status set_last_error(dl_status s, const char* msg);  // dl_host.cu
}

using namespace dl;

namespace {

// 8 MiB: a 512-byte binding slot, a 256-byte status slot, up to 4096
// arrival counters, then the partials (G CTAs x 2 slots x QRp rows x 129
// floats: 128 output dims + the row's log-sum-exp).  At 152 CTAs that holds
// every query-row padding up to 32; 64-row groups need num_sms <= 126.
constexpr size_t kScratchBytes = 8u << 20;
constexpr size_t kBindingOff = 0;
constexpr size_t kStatusOff = 512;
constexpr size_t kCounterOff = 768;
constexpr int kMaxPairs = 4096;
constexpr size_t kPartialOff = kCounterOff + kMaxPairs * sizeof(unsigned);  // 17152
constexpr int kMaxDevices = 64;
constexpr unsigned long long kBudgetNs = 1000000000ull;

static_assert(sizeof(Binding) <= kStatusOff - kBindingOff, "binding slot");
static_assert(sizeof(DevStatus) <= kCounterOff - kStatusOff, "status slot");
static_assert(kPartialOff % 256 == 0, "partials start 256-byte aligned");

// The scratch itself.  Host code only ever sees a stand-in for it: the
// device address comes from cudaGetSymbolAddress at set-up.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSetup {
  bool ready = false;
  unsigned char* scratch = nullptr;
  int sms = 0;
};

std::mutex g_mu;
DeviceSetup g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;

dl_status err(dl_status s, const char* what, cudaError_t e = cudaSuccess) {
  char buf[256];
  if (e != cudaSuccess)
    std::snprintf(buf, sizeof(buf), "dl_attention_noalloc: %s: %s", what, cudaGetErrorString(e));
  else
    std::snprintf(buf, sizeof(buf), "dl_attention_noalloc: %s", what);
  return set_last_error(s, buf);
}

// One-time set-up of the current device: the scratch's device address, the
// attention kernels' shared-memory attribute and the descriptor encoder.
dl_status setup_current_device(DeviceSetup** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return err(DL_ERR_UNSUPPORTED, "device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceSetup& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p) return err(DL_ERR_CUDA, "cudaGetSymbolAddress(scratch)", e);
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return err(DL_ERR_CUDA, "cudaDeviceGetAttribute", e);
    for (int QRp : {16, 32, 64}) {
      e = cudaFuncSetAttribute(attn_kernel(QRp), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               attn_smem_bytes(QRp, attn_mma_stages(QRp)));
      if (e != cudaSuccess) return err(DL_ERR_CUDA, "cudaFuncSetAttribute", e);
    }
    if (!g_enc) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return err(DL_ERR_CUDA, "cuTensorMapEncodeTiled entry point", e);
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.scratch = static_cast<unsigned char*>(p);
    d.ready = true;
  }
  *out = &d;
  return DL_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" dl_status dl_attention_noalloc(const dl_config* c, int layer, const void* q,
                                          const void* kv_pages, const int32_t* block_table,
                                          const int32_t* positions, void* out, float* out_scale,
                                          int check, void* stream) {
  // ---- host checks (before any CUDA call)
  if (!c) return err(DL_ERR_INVALID_ARG, "cfg is NULL");
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_layers <= 0 || c->num_requests <= 0 ||
      c->tokens_per_request <= 0 || c->page_size <= 0 || c->num_pages <= 0 ||
      c->max_pages_per_request <= 0 || c->max_context <= 0)
    return err(DL_ERR_INVALID_ARG, "non-positive size in cfg");
  if (c->head_dim != 128) return err(DL_ERR_UNSUPPORTED, "head_dim must be 128");
  if (c->n_q_heads % c->n_kv_heads) return err(DL_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
  if (layer < 0 || layer >= c->n_layers) return err(DL_ERR_INVALID_ARG, "layer out of range");
  const int M = c->num_requests * c->tokens_per_request;
  if (M > kMaxM) return err(DL_ERR_UNSUPPORTED, "more than 64 tokens per step");
  const int QR = c->tokens_per_request * (c->n_q_heads / c->n_kv_heads);
  if (QR > kMaxQRows) return err(DL_ERR_UNSUPPORTED, "tokens_per_request * group size > 64");
  if (!(c->page_size % kAttnKeys == 0 || kAttnKeys % c->page_size == 0))
    return err(DL_ERR_UNSUPPORTED, "page_size must divide 64 or be a multiple of 64");
  if (static_cast<long long>(c->max_pages_per_request) * c->page_size < c->max_context)
    return err(DL_ERR_INVALID_ARG, "max_pages_per_request * page_size < max_context");
  const bool fp8 = c->weight_dtype == DL_WEIGHT_FP8_E4M3_B128;
  if (!fp8 && c->weight_dtype != DL_WEIGHT_BF16) return err(DL_ERR_INVALID_ARG, "unknown weight_dtype");
  if (!q || !kv_pages || !block_table || !positions || !out || (fp8 && !out_scale))
    return err(DL_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!al16(q) || !al16(kv_pages) || !al16(out) || (reinterpret_cast<uintptr_t>(block_table) & 3) ||
      (reinterpret_cast<uintptr_t>(positions) & 3) || (reinterpret_cast<uintptr_t>(out_scale) & 3))
    return err(DL_ERR_INVALID_ARG, "misaligned tensor pointer");
  const int pairs = c->num_requests * c->n_kv_heads;
  if (pairs > kMaxPairs)
    return err(DL_ERR_UNSUPPORTED, "num_requests * n_kv_heads > 4096 (scratch counters)");

  DeviceSetup* d = nullptr;
  dl_status st = setup_current_device(&d);
  if (st != DL_OK) return st;

  // ---- launch shape: the plans' split rule without their minimum of four
  // blocks a CTA (the documented scratch limit is stated for this count),
  // the plans' stage rule
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.kv = DPtr{nullptr, SLOT_KV, 0, 0};
  a.bt = DPtr{nullptr, SLOT_BT, 0, 0};
  a.pos = DPtr{nullptr, SLOT_POS, 0, 0};
  a.q = q;
  a.out = out;
  a.out_scale = out_scale;
  a.fp8 = fp8 ? 1 : 0;
  a.R = c->num_requests;
  a.T = c->tokens_per_request;
  a.Hq = c->n_q_heads;
  a.Hkv = c->n_kv_heads;
  a.d = c->head_dim;
  a.P = c->page_size;
  a.num_pages = c->num_pages;
  a.max_pages = c->max_pages_per_request;
  a.layer = layer;
  a.QR = QR;
  a.QRp = QR <= 16 ? 16 : (QR <= 32 ? 32 : 64);
  a.NB = (c->max_context + kAttnKeys - 1) / kAttnKeys;
  a.max_ctx = c->max_context;
  const int sms = c->num_sms > 0 ? std::min(c->num_sms, d->sms) : d->sms;
  a.G = attn_ctas(pairs, a.NB, sms);
  if (static_cast<long long>(pairs) * a.NB * a.G >= (1LL << 32))
    return err(DL_ERR_UNSUPPORTED, "num_requests * n_kv_heads * blocks * CTAs >= 2^32");
  a.stages = attn_mma_stages(a.QRp);
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.d)));
  const size_t need = kPartialOff + static_cast<size_t>(a.G) * 2 * a.QRp * 129 * sizeof(float);
  if (need > kScratchBytes) {
    char buf[200];
    std::snprintf(buf, sizeof(buf),
                  "needs %zu bytes of scratch (%d CTAs x %d padded query rows), the static scratch "
                  "holds %zu; lower num_sms",
                  need, a.G, a.QRp, kScratchBytes);
    return err(DL_ERR_UNSUPPORTED, buf);
  }
  unsigned char* s0 = d->scratch;
  a.ws = reinterpret_cast<float*>(s0 + kPartialOff);
  a.pair_cnt = reinterpret_cast<unsigned*>(s0 + kCounterOff);

  // ---- binding table (pointers + TMA descriptor of the cache)
  Binding b;
  std::memset(&b, 0, sizeof(b));
  b.p[SLOT_KV] = const_cast<void*>(kv_pages);
  b.p[SLOT_BT] = const_cast<int32_t*>(block_table);
  b.p[SLOT_POS] = const_cast<int32_t*>(positions);
  const uint64_t rows = static_cast<uint64_t>(c->n_layers) * c->num_pages * 2 * a.Hkv * a.P;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.d), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.d) * 2};
  cuuint32_t boxd[2] = {64, static_cast<cuuint32_t>(std::min(a.P, kAttnKeys))};
  cuuint32_t estr[2] = {1, 1};
  if (g_enc(&b.kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_pages), dims,
            strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return err(DL_ERR_INVALID_ARG, "kv_pages cannot be described by a TMA descriptor");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Binding* db = reinterpret_cast<Binding*>(s0 + kBindingOff);
  DevStatus* ds = reinterpret_cast<DevStatus*>(s0 + kStatusOff);
  cudaError_t e = launch_bind(db, b, s);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "binding upload", e);
  // the status word and the arrival counters must start at zero (the last
  // arriver of a pair resets its counter, but a failed call may leave some
  // raised); the partials are written before they are read
  e = cudaMemsetAsync(s0 + kStatusOff, 0, kPartialOff - kStatusOff, s);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "cudaMemsetAsync(status, counters)", e);

  KernelCtx ctx;
  ctx.binding = db;
  ctx.status = ds;
  ctx.budget_ns = kBudgetNs;
  ctx.op_id = 0;
  void* args[] = {&a, &ctx};
  e = cudaLaunchKernel(attn_kernel(a.QRp), dim3(a.G), dim3(kThreads), args,
                       static_cast<size_t>(attn_smem_bytes(a.QRp, a.stages)), s);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "attention launch", e);
  if (!check) return DL_OK;

  // ---- optional synchronous check of the device status word
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "cudaStreamSynchronize", e);
  DevStatus h;
  e = cudaMemcpy(&h, ds, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return err(DL_ERR_CUDA, "status read", e);
  if (h.code == DERR_NONE) return DL_OK;
  char buf[200];
  std::snprintf(buf, sizeof(buf), "device error %u: cta %u where %u value %u", h.code, h.info[1],
                h.info[2], h.info[3]);
  return err(h.code == DERR_TIMEOUT ? DL_ERR_TIMEOUT
             : h.code == DERR_BOUNDS ? DL_ERR_DEVICE_BOUNDS
                                     : DL_ERR_CUDA,
             buf);
}
