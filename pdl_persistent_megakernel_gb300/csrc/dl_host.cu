// dl_host.cu -- the plan: validation, buffers, TMA descriptors, per-op launch
// lists, graph capture (serial / graph / graph+PDL schedules), megakernel
// queue packing and validation, and the C ABI of include/dl.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "dl.h"
#include "dl_internal.h"
#include "dl_kernels.h"

using namespace dl;

// ------------------------------------------------------------------ errors
static thread_local std::string g_err;

static dl_status fail(dl_status s, const std::string& msg) {
  g_err = msg;
  return s;
}

extern "C" const char* dl_last_error(void) { return g_err.c_str(); }

// Error reporting for the other translation units of the library.
namespace dl {
dl_status set_last_error(dl_status s, const char* msg) { return fail(s, msg); }
}  // namespace dl

#define CK(call)                                                             \
  do {                                                                       \
    cudaError_t e_ = (call);                                                 \
    if (e_ != cudaSuccess)                                                   \
      return fail(DL_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)); \
  } while (0)

// ------------------------------------------------------- tensor map encode
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool load_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                       cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// [rows, K] row-major matrix, boxes of 128 bytes of K by box_rows rows,
// 128-byte swizzle (the tcgen05 K-major canonical layout).
static bool encode_map(CUtensorMap* m, const void* base, bool u8, uint64_t K,
                       uint64_t rows, uint32_t box_rows) {
  const int eb = u8 ? 1 : 2;
  cuuint64_t dims[2] = {K, rows};
  cuuint64_t strides[1] = {K * eb};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(
      m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// -------------------------------------------------------------------- plan
namespace {

struct LaunchOp {
  OpArgs args;
  const void* kernel = nullptr;
  int grid = 0;
  int smem = 0;
  int branch = 0;  // 0 main chain, 1 side branch (DAG lists)
  int cluster = 1; // thread-block cluster size along x (the split norm)
  std::string name;
};

DPtr fixed(void* p) {
  DPtr d;
  d.p = p;
  d.slot = -1;
  d.pad = 0;
  d.offset = 0;
  return d;
}

DPtr bound(int slot, long long offset = 0) {
  DPtr d;
  d.p = nullptr;
  d.slot = slot;
  d.pad = 0;
  d.offset = offset;
  return d;
}

}  // namespace

struct dl_plan {
  dl_config cfg{};
  std::vector<dl_layer_weights> layers;
  int dev = 0, sms = 0, M = 0, Mp = 0, Mrows = 0, H = 0, I = 0, Hq = 0, Hkv = 0, d = 0;
  int L = 0, V = 0, R = 0, T = 0, P = 0;
  bool fp8 = false, full = false, mma = false;
  int pf_units = 4;    // L2 prefetch units per share (DL_L2_PREFETCH_UNITS; 0: off)
  bool attn_tc = true; // standalone attention on tcgen05 (DL_ATTN=mma_sync: mma.sync)
  // Most operand stages a projection / the tcgen05 attention keeps (in
  // flight before its dependency, and in its ring): DL_GEMM_STAGES,
  // DL_ATTN_STAGES.
  int gemm_stages_max = 5, attn_stages_max = 6;
  Instr* d_noop_queues = nullptr;   // [workers][1] NoOps (the empty megakernel)
  // the DAG schedule's fork and join edges programmatic under PDL
  // (DL_DAG_PROGRAMMATIC_EDGES=0: event edges, as in the non-PDL DAG)
  bool dag_prog_edges = true;
  // tcgen05 attention up to 32 query rows: one S-reading warp and four exp
  // warps on the four SM sub-partitions (DL_ATTN_SPLIT_SOFTMAX=0: two
  // alternating softmax warps of sub-partition 0)
  bool split_sm = true;
  // megakernel: attention shares wait on per-head QKV tile events
  // (DL_MEGA_HEAD_EVENTS=0: on the whole projection)
  bool head_events = true;
  // a projection whose output only feeds the next norm leaves its Stream-K
  // fix-up to that norm (EPI_PARTIALS)
  bool defer_fixup = true;
  // K/V blocks the attention loads before its dependency wait (0: every
  // block without this step's new keys, up to the ring).  Three measured
  // about 0.6 us faster than the whole ring on the Qwen3-8B FP8 layer at
  // M = 16, context 8192: the early loads compete with the QKV projection
  // still streaming its weights.
  int attn_pre_stages = 3;
  // the tcgen05 attention loads a 64-key block as one 4-D TMA box
  bool attn_kv4 = true;
  // 64-key blocks each attention CTA takes at least (when its pair has them)
  int attn_min_blocks = 4;
  // add + RMSNorm rows split over clusters of up to this many CTAs (1, 2, 4)
  int norm_split = 4;
  unsigned long long budget_ns = 1000000000ull;

  std::vector<void*> allocs;
  Binding* d_binding = nullptr;
  DevStatus* d_status = nullptr;
  unsigned long long* d_trace = nullptr;  // trace build: [trace_ops][sms][kTraceSlots]
  int trace_ops = 0;
  void *h1 = nullptr, *attn = nullptr, *h2 = nullptr, *act = nullptr;
  float *h1s = nullptr, *attns = nullptr, *h2s = nullptr, *acts = nullptr;
  void *r1 = nullptr, *r2 = nullptr, *o2 = nullptr, *y = nullptr, *q = nullptr;
  void *hfin = nullptr, *rfin = nullptr;
  float* logits = nullptr;
  float* best_val = nullptr;
  int* best_idx = nullptr;
  float* rope = nullptr;
  float* ws_gemm[2] = {nullptr, nullptr};
  float* ws_attn = nullptr;
  unsigned* counters = nullptr;
  size_t n_counters = 0;
  CUtensorMap* d_maps = nullptr;
  std::vector<CUtensorMap> h_maps;

  std::vector<LaunchOp> lin, dag;
  // the megakernel's ops: the linear list with every Stream-K fix-up in its
  // projection (its norm instructions run on M workers, where reading the
  // projection's partials measured slower than the fix-up on all of them)
  std::vector<LaunchOp> mega;

  // megakernel
  OpArgs* d_ops = nullptr;
  Instr* d_queues = nullptr;
  unsigned* d_events = nullptr;
  unsigned* d_finish = nullptr;
  std::vector<Instr> queues;
  int qlen = 0, workers = 0, n_events = 0, mega_smem = 0;
  int mega_ns = 0, mega_slot = 0, mega_priv_off = 0;

  cudaGraphExec_t exec[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  cudaStream_t cap = nullptr, side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;

  Binding last{};
  bool have_last = false;
  int perturb_idx = -1;      // instruction whose wait the failure test raised
  unsigned perturb_orig = 0;

  // end-to-end staging
  void *st_x = nullptr, *st_res = nullptr, *st_out = nullptr;
  int *st_bt = nullptr, *st_pos = nullptr;
};

static dl_status dev_alloc(dl_plan* p, void** out, size_t bytes) {
  void* ptr = nullptr;
  if (bytes == 0) bytes = 16;
  const cudaError_t e = cudaMalloc(&ptr, bytes);
  if (e != cudaSuccess)
    return fail(DL_ERR_OOM, std::string("cudaMalloc: ") + cudaGetErrorString(e));
  p->allocs.push_back(ptr);
  if (cudaMemset(ptr, 0, bytes) != cudaSuccess) return fail(DL_ERR_CUDA, "cudaMemset");
  *out = ptr;
  return DL_OK;
}

template <typename T>
static dl_status dalloc(dl_plan* p, T** out, size_t bytes) {
  void* v = nullptr;
  const dl_status s = dev_alloc(p, &v, bytes);
  *out = static_cast<T*>(v);
  return s;
}

static void free_plan(dl_plan* p) {
  if (!p) return;
  for (auto& e : p->exec)
    if (e) cudaGraphExecDestroy(e);
  if (p->cap) cudaStreamDestroy(p->cap);
  if (p->side) cudaStreamDestroy(p->side);
  if (p->d_noop_queues) cudaFree(p->d_noop_queues);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  for (void* a : p->allocs) cudaFree(a);
  delete p;
}

static KernelCtx make_ctx(const dl_plan* p, int op_id) {
  KernelCtx c;
  c.binding = p->d_binding;
  c.status = p->d_status;
  c.budget_ns = p->budget_ns;
  c.op_id = op_id;
  c.trace = p->d_trace;
  c.trace_ctas = p->sms;
  return c;
}

// ------------------------------------------------------------ op builders
constexpr int kGemmSmemTarget = 210 * 1024;
constexpr int kAttnTcSmemTarget = 224 * 1024;
static int choose_stages(int stage_bytes, int fixed_bytes, int target) {
  int s = (target - fixed_bytes) / stage_bytes;
  return std::max(2, std::min(kMaxStages, s));
}

static LaunchOp make_norm(dl_plan* p, DPtr x, DPtr res, DPtr rout, const void* w, void* hout,
                          float* hscale, bool fp8, const char* name) {
  LaunchOp op;
  std::memset(&op.args, 0, sizeof(op.args));
  op.args.kind = OP_NORM;
  NormArgs& a = op.args.norm;
  a.x = x;
  a.res = res;
  a.r_out = rout;
  a.w = w;
  a.h_out = hout;
  a.h_scale = hscale;
  a.fp8 = fp8 ? 1 : 0;
  a.M = p->M;
  a.H = p->H;
  a.rows_per_cta = 1;
  a.eps = p->cfg.eps;
  // a row over a cluster of 4 (or 2) CTAs: a part is a whole number of
  // 128-column quantisation groups and tiles, and all rows' clusters fit in
  // one wave (the megakernel runs one share per worker)
  int split = 1;
  for (int k : {4, 2})
    if (split == 1 && k <= p->norm_split && p->H % (k * 128) == 0 && p->H / k <= 2048 &&
        p->M * k <= p->sms)
      split = k;
  op.kernel = norm_kernel(p->H, split);
  op.grid = p->M * split;
  op.cluster = split;
  a.split = split;
  op.smem = norm_smem_bytes();
  op.name = name;
  return op;
}

struct GemmSpec {
  const CUtensorMap* tw;
  const CUtensorMap* tx;
  const float* wscale;
  const float* xscale;
  bool fp8;
  int K;
  int NT;
  int t_base;
  bool pair;
  int up_row;
  int epi;
  int ws_slot;
  const char* name;
};

static LaunchOp make_gemm(dl_plan* p, const GemmSpec& s, unsigned* cnt) {
  LaunchOp op;
  std::memset(&op.args, 0, sizeof(op.args));
  op.args.kind = OP_GEMM;
  GemmArgs& a = op.args.gemm;
  a.tmap_w = s.tw;
  a.tmap_x = s.tx;
  a.w_scale = s.wscale;
  a.x_scale = s.xscale;
  a.fp8 = s.fp8 ? 1 : 0;
  a.mma = p->mma ? 1 : 0;
  a.M = p->M;
  a.Mp = p->mma ? p->Mp : p->M;
  a.K = s.K;
  a.KB = s.K * (s.fp8 ? 1 : 2) / 128;
  a.NT = s.NT;
  a.t_base = s.t_base;
  a.pair = s.pair ? 1 : 0;
  a.up_row = s.up_row;
  const long long U = static_cast<long long>(a.NT) * a.KB;
  a.G = static_cast<int>(std::min<long long>(p->sms, U));
  a.share_max = static_cast<int>((U + a.G - 1) / a.G);
  const int npair = s.pair ? 2 : 1;
  // a stage: 32 KiB of tiles (gate + up, or two consecutive units) and one
  // activation slice per unit
  const int stage_bytes = 32768 + (npair == 1 ? 2 : 1) * (((a.Mp * 128 + 1023) / 1024) * 1024);
  const int fixed_bytes = gemm_smem_bytes(npair, a.Mp, 0, a.KB, a.fp8, s.epi, a.M, a.share_max);
  // one CTA per SM; 3-4 stages of 32 KiB in flight per SM already reach the
  // HBM copy rate, a few more absorb jitter
  a.stages = std::min(p->gemm_stages_max, choose_stages(stage_bytes, fixed_bytes, kGemmSmemTarget));
  a.tmem_bufs = a.mma ? std::min(4, 512 / (npair * a.Mp)) : 1;
  a.epi = s.epi;
  a.ws = p->ws_gemm[s.ws_slot];
  a.tile_cnt = cnt;
  a.done_cnt = cnt + a.NT;
  op.kernel = gemm_kernel(a.mma, a.mma ? a.Mp : a.M);
  op.grid = a.G;
  op.smem = gemm_smem_bytes(npair, a.Mp, a.stages, a.KB, a.fp8, s.epi, a.M, a.share_max);
  op.name = s.name;
  return op;
}

// Deferred Stream-K fix-up: a bf16-output projection directly followed by a
// norm that reads exactly that output (the O projection before the second
// norm, the down projection before the next layer's first norm or the final
// norm) skips its fix-up and epilogue: each CTA writes the partial of every
// tile its range touches and leaves, and the norm forms each element as the
// CTA-ordered sum of the tile's partials (the order of the fix-up, so the
// result is the same to the bit) before its residual add.  The projection's
// tail -- waiting for the other contributors, reading their partials, the
// epilogue -- leaves the critical path; the norm reads the partials in the
// round trip in which it read the projection's output.  Taken only when
// every CTA's range touches at most two tiles (its two partial slots) and no
// tile has more than kMaxPartContrib contributors.
static unsigned host_sk_begin(unsigned U, int G, int c);
static void defer_fixups(std::vector<LaunchOp>& ops) {
  for (size_t i = 0; i + 1 < ops.size(); ++i) {
    LaunchOp& g = ops[i];
    LaunchOp& n = ops[i + 1];
    if (g.args.kind != OP_GEMM || n.args.kind != OP_NORM || g.branch != 0 || n.branch != 0) continue;
    GemmArgs& a = g.args.gemm;
    NormArgs& na = n.args.norm;
    if (a.epi != EPI_STORE_BF16 || a.pair || a.t_base != 0 || a.NT * 128 != na.H ||
        a.out.slot >= 0 || a.out.p != na.x.p || a.out.offset != na.x.offset || a.ldo != na.H ||
        na.x.slot >= 0 || na.H > 64 * 128)
      continue;
    const unsigned U = static_cast<unsigned>(a.NT) * static_cast<unsigned>(a.KB);
    bool ok = true;
    std::vector<int> contrib(static_cast<size_t>(a.NT), 0);
    for (int c = 0; c < a.G && ok; ++c) {
      const unsigned u0 = host_sk_begin(U, a.G, c), u1 = host_sk_begin(U, a.G, c + 1);
      if (u1 <= u0) continue;
      const int t0 = static_cast<int>(u0 / a.KB), t1 = static_cast<int>((u1 - 1) / a.KB);
      if (t1 - t0 > 1) ok = false;
      for (int t = t0; t <= t1 && ok; ++t)
        if (++contrib[t] > kMaxPartContrib) ok = false;
    }
    if (!ok) continue;
    a.epi = EPI_PARTIALS;
    na.part = a.ws;
    na.part_U = static_cast<int>(U);
    na.part_G = a.G;
    na.part_KB = a.KB;
    na.part_mp = a.Mp;
  }
}

// CTAs of the split-KV attention: a whole number of CTAs per (request, kv
// head) pair when the pairs are fewer than the SMs, so that no CTA's range
// straddles two pairs (a straddling CTA merges and publishes mid-range and
// holds up both pairs' combines); at most 62 per pair (the combine's weights
// sit in two lanes of a warp); never more than the units.  min_blocks > 1
// gives each CTA at least that many 64-key blocks of its pair (fewer
// contributors for the pair's combine).
int dl::attn_ctas(int pairs, int nb, int sms, int min_blocks) {
  const long long U = static_cast<long long>(pairs) * nb;
  const int per = std::min(std::min(62, sms / std::max(1, pairs)),
                           std::max(1, (nb + min_blocks - 1) / std::max(1, min_blocks)));
  long long g = pairs <= sms ? static_cast<long long>(pairs) * per : sms;
  return static_cast<int>(std::max(1LL, std::min(g, U)));
}

// 4 stages of 32 KiB keep the mma.sync engine fed (more add nothing).
int dl::attn_mma_stages(int QRp) {
  return std::max(2, std::min(4, (kGemmSmemTarget - attn_smem_bytes(QRp, 0)) / (4 * kAttnKeys * 128)));
}

static LaunchOp make_attn(dl_plan* p, int layer, unsigned* cnt) {
  LaunchOp op;
  std::memset(&op.args, 0, sizeof(op.args));
  op.args.kind = OP_ATTN;
  AttnArgs& a = op.args.attn;
  a.kv = bound(SLOT_KV);
  a.bt = bound(SLOT_BT);
  a.pos = bound(SLOT_POS);
  a.q = p->q;
  a.out = p->attn;
  a.out_scale = p->attns;
  a.fp8 = p->fp8 ? 1 : 0;
  a.R = p->R;
  a.T = p->T;
  a.Hq = p->Hq;
  a.Hkv = p->Hkv;
  a.d = p->d;
  a.P = p->P;
  a.num_pages = p->cfg.num_pages;
  a.max_pages = p->cfg.max_pages_per_request;
  a.layer = layer;
  a.QR = p->T * (p->Hq / p->Hkv);
  a.QRp = a.QR <= 16 ? 16 : (a.QR <= 32 ? 32 : 64);
  a.NB = (p->cfg.max_context + kAttnKeys - 1) / kAttnKeys;
  a.max_ctx = p->cfg.max_context;
  a.pre_stages = p->attn_pre_stages;
  a.kv4 = p->attn_tc && p->attn_kv4 && p->P % kAttnKeys == 0 && p->d == 128 ? 1 : 0;
  a.split_sm = p->split_sm ? 1 : 0;
  a.G = attn_ctas(a.R * a.Hkv, a.NB, p->sms, p->attn_min_blocks);
  // stages of 32 KiB: the tcgen05 engine holds a block from its arrival to
  // its PV commit, so it takes as many as fit (up to 6)
  a.stages = p->attn_tc
      ? std::max(2, std::min(p->attn_stages_max, (kAttnTcSmemTarget - attn_tc_smem_bytes(a.QRp, 0)) /
                                    (4 * kAttnKeys * 128)))
      : attn_mma_stages(a.QRp);
  a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(p->d)));
  a.ws = p->ws_attn;
  a.pair_cnt = cnt;
  op.kernel = p->attn_tc ? attn_tc_kernel() : attn_kernel(a.QRp);
  op.grid = a.G;
  op.smem = p->attn_tc ? attn_tc_smem_bytes(a.QRp, a.stages) : attn_smem_bytes(a.QRp, a.stages);
  op.name = "attention";
  return op;
}

// ------------------------------------------------------------ validation
static dl_status check_config(const dl_config* c) {
  if (!c) return fail(DL_ERR_INVALID_ARG, "cfg is NULL");
  if (c->hidden <= 0 || c->inter <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 ||
      c->n_layers <= 0 || c->num_requests <= 0 || c->tokens_per_request <= 0 ||
      c->page_size <= 0 || c->num_pages <= 0 || c->max_pages_per_request <= 0 ||
      c->max_context <= 0 || c->vocab < 0)
    return fail(DL_ERR_INVALID_ARG, "non-positive size in cfg");
  if (c->head_dim != 128) return fail(DL_ERR_UNSUPPORTED, "head_dim must be 128");
  if (c->n_q_heads % c->n_kv_heads) return fail(DL_ERR_INVALID_ARG, "n_q_heads % n_kv_heads != 0");
  if (c->hidden % 128 || c->inter % 128) return fail(DL_ERR_UNSUPPORTED, "hidden and inter must be multiples of 128");
  if (c->hidden > 8192) return fail(DL_ERR_UNSUPPORTED, "hidden > 8192");
  if (c->vocab % 128) return fail(DL_ERR_UNSUPPORTED, "vocab must be a multiple of 128");
  const int M = c->num_requests * c->tokens_per_request;
  if (M > kMaxM) return fail(DL_ERR_UNSUPPORTED, "more than 64 tokens per step");
  const int QR = c->tokens_per_request * (c->n_q_heads / c->n_kv_heads);
  if (QR > kMaxQRows) return fail(DL_ERR_UNSUPPORTED, "tokens_per_request * group size > 64");
  if (!(c->page_size % kAttnKeys == 0 || kAttnKeys % c->page_size == 0))
    return fail(DL_ERR_UNSUPPORTED, "page_size must divide 64 or be a multiple of 64");
  if (static_cast<long long>(c->max_pages_per_request) * c->page_size < c->max_context)
    return fail(DL_ERR_INVALID_ARG, "max_pages_per_request * page_size < max_context");
  if (c->weight_dtype != DL_WEIGHT_BF16 && c->weight_dtype != DL_WEIGHT_FP8_E4M3_B128)
    return fail(DL_ERR_INVALID_ARG, "unknown weight_dtype");
  if (c->weight_dtype == DL_WEIGHT_FP8_E4M3_B128 && c->vocab)
    return fail(DL_ERR_UNSUPPORTED, "FP8 weights are supported for layer plans");
  if (!c->layers) return fail(DL_ERR_INVALID_ARG, "layers is NULL");
  return DL_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ------------------------------------------------- graph / launch helpers
// prog_event: the launch also records a programmatic event, which fires
// once every CTA of the kernel has passed griddepcontrol.launch_dependents
// (not at block start): a launch on another stream that waits on it is the
// kernel's programmatic dependent, as the next launch on the same stream is.
static cudaError_t launch_op(const dl_plan* p, const LaunchOp& op, cudaStream_t s, bool pdl,
                             int op_id, cudaEvent_t prog_event = nullptr) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(op.grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = op.smem;
  lc.stream = s;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (prog_event) {
    attr[lc.numAttrs].id = cudaLaunchAttributeProgrammaticEvent;
    attr[lc.numAttrs].val.programmaticEvent.event = prog_event;
    attr[lc.numAttrs].val.programmaticEvent.flags = 0;
    attr[lc.numAttrs].val.programmaticEvent.triggerAtBlockStart = 0;
    ++lc.numAttrs;
  }
  if (op.cluster > 1) {
    attr[lc.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[lc.numAttrs].val.clusterDim.x = static_cast<unsigned>(op.cluster);
    attr[lc.numAttrs].val.clusterDim.y = 1;
    attr[lc.numAttrs].val.clusterDim.z = 1;
    ++lc.numAttrs;
  }
  KernelCtx ctx = make_ctx(p, op_id);
  switch (op.args.kind) {
    case OP_NORM: {
      NormArgs a = op.args.norm;
      void* args[] = {&a, &ctx};
      return cudaLaunchKernelExC(&lc, op.kernel, args);
    }
    case OP_GEMM: {
      GemmArgs a = op.args.gemm;
      void* args[] = {&a, &ctx};
      return cudaLaunchKernelExC(&lc, op.kernel, args);
    }
    case OP_ATTN: {
      AttnArgs a = op.args.attn;
      void* args[] = {&a, &ctx};
      return cudaLaunchKernelExC(&lc, op.kernel, args);
    }
    default:
      return cudaErrorInvalidValue;
  }
}

// The DAG schedule's branch: op i with branch == 1 runs on the side stream,
// forked after the main stream's previous op; the next op with branch == 2
// joins it.  Under programmatic launch both edges are programmatic: the fork
// op and the branch op record programmatic events (fired when all their
// CTAs have passed launch_dependents), so the branch op's CTAs may start,
// and the joining op's may run their prologue and weight / K/V prefetch,
// before their producers finish; every kernel still waits for its
// producers' completion (griddepcontrol.wait) before a dependent read.
// Without it the edges are full event dependencies.
static cudaError_t enqueue_list(dl_plan* p, const std::vector<LaunchOp>& ops, cudaStream_t s,
                                bool pdl) {
  const bool prog = pdl && p->dag_prog_edges;
  for (size_t i = 0; i < ops.size(); ++i) {
    const LaunchOp& op = ops[i];
    const bool forks = i + 1 < ops.size() && ops[i + 1].branch == 1;
    if (op.branch == 1) {
      // side branch: forks from the main stream after the previous main op
      cudaError_t e;
      if (!prog) {
        e = cudaEventRecord(p->ev_fork, s);
        if (e != cudaSuccess) return e;
      }
      e = cudaStreamWaitEvent(p->side, p->ev_fork, 0);
      if (e != cudaSuccess) return e;
      e = launch_op(p, op, p->side, pdl, static_cast<int>(i), prog ? p->ev_join : nullptr);
      if (e != cudaSuccess) return e;
      if (!prog) {
        e = cudaEventRecord(p->ev_join, p->side);
        if (e != cudaSuccess) return e;
      }
      continue;
    }
    if (op.branch == 2) {
      // join point: the main stream waits for the side branch first
      cudaError_t e = cudaStreamWaitEvent(s, p->ev_join, 0);
      if (e != cudaSuccess) return e;
    }
    const cudaError_t e =
        launch_op(p, op, s, pdl, static_cast<int>(i), (prog && forks) ? p->ev_fork : nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

static dl_status capture_graph(dl_plan* p, int mode) {
  const bool dag = (mode == DL_MODE_PDL_GRAPH || mode == DL_MODE_GRAPH_DAG);
  const bool pdl = (mode == DL_MODE_PDL_GRAPH || mode == DL_MODE_GRAPH_LINEAR_PDL);
  const std::vector<LaunchOp>& ops = dag ? p->dag : p->lin;
  cudaGraph_t g = nullptr;
  CK(cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal));
  const cudaError_t e = enqueue_list(p, ops, p->cap, pdl);
  const cudaError_t e2 = cudaStreamEndCapture(p->cap, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return fail(DL_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(e));
  }
  if (e2 != cudaSuccess) return fail(DL_ERR_CUDA, std::string("end capture: ") + cudaGetErrorString(e2));
  const cudaError_t e3 = cudaGraphInstantiate(&p->exec[mode], g, 0);
  cudaGraphDestroy(g);
  if (e3 != cudaSuccess) return fail(DL_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(e3));
  return DL_OK;
}

// ------------------------------------------------------------ megakernel
// Instructions of op k run on workers 0 .. G_k - 1; every instruction of op k
// waits until event k-1 (one count per finished instruction of op k-1)
// reaches G_{k-1}, and adds 1 to event k when done.  The ops are listed in a
// topological order in which each depends on its predecessor, so the chain
// of waits orders every true dependency (and every write-after-read reuse
// of a buffer) of the list.
// The device's Stream-K range arithmetic (32-bit, as in the kernels).
static unsigned host_sk_begin(unsigned U, int G, int c) {
  return (U * static_cast<unsigned>(c)) / static_cast<unsigned>(G);
}
static int host_sk_owner(unsigned U, int G, unsigned x) {
  int c = static_cast<int>((x * static_cast<unsigned>(G)) / U);
  if (c >= G) c = G - 1;
  while (c > 0 && host_sk_begin(U, G, c) > x) --c;
  while (c + 1 < G && host_sk_begin(U, G, c + 1) <= x) ++c;
  return c;
}

static dl_status build_mega(dl_plan* p) {
  const std::vector<LaunchOp>& ops = p->mega;
  const int nops = static_cast<int>(ops.size());
  p->workers = p->sms;
  std::vector<std::vector<Instr>> qs(p->workers);
  for (int k = 0; k < nops; ++k) {
    const int G = ops[k].grid;
    if (G > p->workers) return fail(DL_ERR_PLAN_INVALID, "op wider than the worker grid");
    for (int c = 0; c < G; ++c) {
      Instr in;
      std::memset(&in, 0, sizeof(in));
      in.op_row = static_cast<uint32_t>(k);
      in.cta = static_cast<uint32_t>(c);
      if (k > 0) {
        in.n_wait = 1;
        in.wait_event[0] = static_cast<uint32_t>(k - 1);
        in.wait_value[0] = static_cast<uint32_t>(ops[k - 1].grid);
      }
      in.n_signal = 1;
      in.signal_event[0] = static_cast<uint32_t>(k);
      in.signal_inc[0] = 1;
      qs[c].push_back(in);
    }
  }
  // Per-head events (the per-head events of page "Kernel-Mega-PDL",
  // section 4, where a downstream task waits only on the heads it reads):
  // an attention share waits for the QKV tiles of the kv heads of its
  // (request, kv head) pairs -- the group's q heads, its k head and its v
  // head -- instead of the whole projection.  A tile is finished (Stream-K
  // fix-up and epilogue) by the share that owns its first unit, so that
  // share's instruction adds 1 to the tile's head event when it ends.
  int n_events = nops;
  if (p->head_events) {
    for (int k = 1; k < nops; ++k) {
      const LaunchOp& at = ops[k];
      const LaunchOp& qk = ops[k - 1];
      if (at.args.kind != OP_ATTN || qk.args.kind != OP_GEMM ||
          qk.args.gemm.epi != EPI_QKV_ROPE)
        continue;
      const GemmArgs& g = qk.args.gemm;
      const AttnArgs& a = at.args.attn;
      const int grp_size = a.Hq / a.Hkv;
      if (g.t_base != 0 || g.NT != a.Hq + 2 * a.Hkv) continue;
      const int ev0 = n_events;
      n_events += a.Hkv;
      const unsigned U = static_cast<unsigned>(g.NT) * static_cast<unsigned>(g.KB);
      for (int t = 0; t < g.NT; ++t) {
        const int h = t < a.Hq ? t / grp_size : (t < a.Hq + a.Hkv ? t - a.Hq : t - a.Hq - a.Hkv);
        const int own = host_sk_owner(U, g.G, static_cast<unsigned>(t) * g.KB);
        Instr* in = nullptr;
        for (Instr& x : qs[own])
          if (x.op_row == static_cast<uint32_t>(k - 1)) in = &x;
        if (!in) return fail(DL_ERR_PLAN_INVALID, "tile owner without a QKV instruction");
        bool merged = false;
        for (uint32_t sgi = 0; sgi < in->n_signal; ++sgi)
          if (instr_signal_event(*in, sgi) == static_cast<uint32_t>(ev0 + h)) {
            (sgi < 2 ? in->signal_inc[sgi] : in->signal_inc_hi[sgi - 2]) += 1;
            merged = true;
          }
        if (!merged) {
          if (in->n_signal >= kMaxSignals)
            return fail(DL_ERR_PLAN_INVALID, "a QKV share finishes tiles of too many heads");
          const uint32_t sgi = in->n_signal++;
          if (sgi < 2) {
            in->signal_event[sgi] = static_cast<uint32_t>(ev0 + h);
            in->signal_inc[sgi] = 1;
          } else {
            in->signal_event_hi[sgi - 2] = static_cast<uint32_t>(ev0 + h);
            in->signal_inc_hi[sgi - 2] = 1;
          }
        }
      }
      // each attention share: the head events of its pairs (at most four
      // distinct heads; otherwise it keeps the wait on the whole projection)
      const unsigned Ua = static_cast<unsigned>(a.R * a.Hkv) * static_cast<unsigned>(a.NB);
      for (int c = 0; c < at.grid; ++c) {
        const unsigned u0 = host_sk_begin(Ua, a.G, c), u1 = host_sk_begin(Ua, a.G, c + 1);
        if (u1 <= u0) continue;
        int heads[4], nh = 0;
        bool too_many = false;
        for (unsigned pr = u0 / a.NB; pr <= (u1 - 1) / a.NB && !too_many; ++pr) {
          const int h = static_cast<int>(pr % a.Hkv);
          bool seen = false;
          for (int i = 0; i < nh; ++i) seen |= heads[i] == h;
          if (seen) continue;
          if (nh == 4) too_many = true;
          else heads[nh++] = h;
        }
        if (too_many) continue;
        Instr* in = nullptr;
        for (Instr& x : qs[c])
          if (x.op_row == static_cast<uint32_t>(k)) in = &x;
        if (!in) return fail(DL_ERR_PLAN_INVALID, "attention share without an instruction");
        in->n_wait = static_cast<uint32_t>(nh);
        for (int i = 0; i < nh; ++i) {
          in->wait_event[i] = static_cast<uint32_t>(ev0 + heads[i]);
          in->wait_value[i] = static_cast<uint32_t>(grp_size + 2);
        }
      }
    }
  }
  p->qlen = 0;
  for (auto& q : qs) p->qlen = std::max<int>(p->qlen, static_cast<int>(q.size()));
  p->qlen += 1;  // at least one NoOp terminator per queue
  p->queues.assign(static_cast<size_t>(p->workers) * p->qlen, Instr{});
  for (int w = 0; w < p->workers; ++w)
    for (int i = 0; i < p->qlen; ++i) {
      Instr& dst = p->queues[static_cast<size_t>(w) * p->qlen + i];
      if (i < static_cast<int>(qs[w].size())) {
        dst = qs[w][i];
      } else {
        std::memset(&dst, 0, sizeof(dst));
        dst.op_row = 0xffffffffu;
      }
    }
  p->n_events = n_events;
  return DL_OK;
}

// Host validator: every wait names an event of an earlier op whose total
// signals reach the threshold, and every queue is in global op order with
// its NoOp terminator last.  Returns DL_ERR_PLAN_INVALID with a message
// otherwise.
static dl_status validate_queues(const Instr* queues, int workers, int qlen, int n_events) {
  // per event: the total of its signals and the latest op that signals it
  std::vector<unsigned long long> total(static_cast<size_t>(n_events), 0);
  std::vector<long long> last_producer(static_cast<size_t>(n_events), -1);
  const size_t n = static_cast<size_t>(workers) * qlen;
  for (size_t i = 0; i < n; ++i) {
    const Instr& in = queues[i];
    if (in.op_row == 0xffffffffu) continue;
    if (in.n_wait > kMaxWaits || in.n_signal > kMaxSignals)
      return fail(DL_ERR_PLAN_INVALID, "too many waits/signals");
    for (uint32_t s = 0; s < in.n_signal; ++s) {
      const uint32_t e = instr_signal_event(in, s);
      if (e >= static_cast<uint32_t>(n_events))
        return fail(DL_ERR_PLAN_INVALID, "signal of an unknown event");
      total[e] += instr_signal_inc(in, s);
      last_producer[e] = std::max<long long>(last_producer[e], in.op_row);
    }
  }
  for (int w = 0; w < workers; ++w) {
    long long prev = -1;
    bool ended = false;
    for (int i = 0; i < qlen; ++i) {
      const Instr& in = queues[static_cast<size_t>(w) * qlen + i];
      if (in.op_row == 0xffffffffu) {
        ended = true;
        continue;
      }
      if (ended) return fail(DL_ERR_PLAN_INVALID, "instruction after the NoOp terminator");
      if (static_cast<long long>(in.op_row) <= prev)
        return fail(DL_ERR_PLAN_INVALID, "queue not in global op order");
      prev = in.op_row;
      for (uint32_t k = 0; k < in.n_wait; ++k) {
        const uint32_t e = in.wait_event[k];
        if (e >= static_cast<uint32_t>(n_events))
          return fail(DL_ERR_PLAN_INVALID, "wait on an unknown event");
        // every instruction that signals e must come earlier in the global
        // order; then the earliest unfinished instruction can always run
        if (last_producer[e] >= static_cast<long long>(in.op_row))
          return fail(DL_ERR_PLAN_INVALID, "wait on an event of a later op (deadlock)");
        if (in.wait_value[k] > total[e])
          return fail(DL_ERR_PLAN_INVALID, "wait threshold above the event's total signals");
      }
    }
    if (!ended) return fail(DL_ERR_PLAN_INVALID, "queue without its NoOp terminator");
  }
  return DL_OK;
}

static dl_status validate_mega(const dl_plan* p) {
  return validate_queues(p->queues.data(), p->workers, p->qlen, p->n_events);
}

static dl_status upload_mega(dl_plan* p) {
  CK(cudaMemcpy(p->d_queues, p->queues.data(), p->queues.size() * sizeof(Instr),
                cudaMemcpyHostToDevice));
  return DL_OK;
}

static cudaError_t launch_mega(dl_plan* p, cudaStream_t s) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(p->workers);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = p->mega_smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  MegaArgs m;
  m.ops = p->d_ops;
  m.queues = p->d_queues;
  m.qlen = p->qlen;
  m.workers = p->workers;
  m.events = p->d_events;
  m.finish_cnt = p->d_finish;
  m.num_events = p->n_events;
  m.budget_ns = p->budget_ns;
  m.trace = nullptr;
  m.ns = p->mega_ns;
  m.slot_bytes = p->mega_slot;
  m.priv_off = p->mega_priv_off;
  KernelCtx ctx = make_ctx(p, -1);
  void* args[] = {&m, &ctx};
  return cudaLaunchKernelExC(&lc, mega_kernel(), args);
}

// The megakernel with every worker's queue a single NoOp: the framework's
// own cost (launch of the persistent grid, barrier and TMEM set-up, the
// queue read, the counters' reset by the last worker, teardown).
extern "C" dl_status dl_plan_bench_empty_megakernel(dl_plan* p, int iters, double* us_per_launch,
                                                    void* stream) {
  if (!p || !us_per_launch || iters < 1) return fail(DL_ERR_INVALID_ARG, "NULL plan or output");
  if (!p->d_queues) return fail(DL_ERR_INVALID_ARG, "no megakernel plan");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!p->d_noop_queues) {
    std::vector<Instr> noop(static_cast<size_t>(p->workers));
    for (Instr& in : noop) {
      std::memset(&in, 0, sizeof(in));
      in.op_row = 0xffffffffu;
    }
    CK(cudaMalloc(&p->d_noop_queues, noop.size() * sizeof(Instr)));
    CK(cudaMemcpy(p->d_noop_queues, noop.data(), noop.size() * sizeof(Instr),
                  cudaMemcpyHostToDevice));
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(p->workers);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = p->mega_smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  MegaArgs m;
  std::memset(&m, 0, sizeof(m));
  m.ops = p->d_ops;
  m.queues = p->d_noop_queues;
  m.qlen = 1;
  m.workers = p->workers;
  m.events = p->d_events;
  m.finish_cnt = p->d_finish;
  m.num_events = p->n_events;
  m.budget_ns = p->budget_ns;
  m.trace = nullptr;
  m.ns = p->mega_ns;
  m.slot_bytes = p->mega_slot;
  m.priv_off = p->mega_priv_off;
  KernelCtx ctx = make_ctx(p, -1);
  void* args[] = {&m, &ctx};
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  CK(cudaLaunchKernelExC(&lc, mega_kernel(), args));   // warm-up
  CK(cudaEventRecord(e0, s));
  for (int i = 0; i < iters; ++i) CK(cudaLaunchKernelExC(&lc, mega_kernel(), args));
  CK(cudaEventRecord(e1, s));
  CK(cudaEventSynchronize(e1));
  float ms = 0.f;
  CK(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *us_per_launch = 1e3 * ms / iters;
  return DL_OK;
}

// ------------------------------------------------------------- creation
static dl_status build_plan(dl_plan* p) {
  const dl_config& c = p->cfg;
  CK(cudaGetDevice(&p->dev));
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->dev));
  p->sms = c.num_sms > 0 ? std::min(c.num_sms, sms) : sms;
  p->H = c.hidden;
  p->I = c.inter;
  p->Hq = c.n_q_heads;
  p->Hkv = c.n_kv_heads;
  p->d = c.head_dim;
  p->L = c.n_layers;
  p->V = c.vocab;
  p->R = c.num_requests;
  p->T = c.tokens_per_request;
  p->P = c.page_size;
  p->M = p->R * p->T;
  p->fp8 = c.weight_dtype == DL_WEIGHT_FP8_E4M3_B128;
  p->full = c.vocab > 0;
  // One token: the CUDA-core GEMV (a warp per 16 rows).  From two tokens on,
  // tcgen05 with the tokens padded to N = 16: at 4 tokens the GEMV is bound
  // by its FP8 unpacking and dot products (measured 1.05 us per unit of the
  // Qwen3-8B QKV projection, against 0.41 us for tcgen05 at 16 tokens).
  p->mma = p->M > 1;
  p->Mp = p->mma ? (p->M <= 16 ? 16 : (p->M <= 32 ? 32 : 64)) : p->M;
  p->Mrows = p->Mp;
  if (!load_encode()) return fail(DL_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");

  const int H = p->H, I = p->I, M = p->M, Mr = p->Mrows, QD = p->Hq * p->d;
  const size_t eb = p->fp8 ? 1 : 2;
  dl_status s;
#define DA(ptr, bytes)                       \
  if ((s = dalloc(p, &(ptr), (bytes))) != DL_OK) return s;
  DA(p->d_binding, sizeof(Binding));
  DA(p->d_status, sizeof(DevStatus));
  DA(p->h1, static_cast<size_t>(Mr) * H * eb);
  DA(p->h2, static_cast<size_t>(Mr) * H * eb);
  DA(p->attn, static_cast<size_t>(Mr) * QD * eb);
  DA(p->act, static_cast<size_t>(Mr) * I * eb);
  DA(p->h1s, static_cast<size_t>(M) * (H / 128) * 4);
  DA(p->h2s, static_cast<size_t>(M) * (H / 128) * 4);
  DA(p->attns, static_cast<size_t>(M) * (QD / 128) * 4);
  DA(p->acts, static_cast<size_t>(M) * (I / 128) * 4);
  DA(p->r1, static_cast<size_t>(M) * H * 2);
  DA(p->r2, static_cast<size_t>(M) * H * 2);
  DA(p->o2, static_cast<size_t>(M) * H * 2);
  DA(p->y, static_cast<size_t>(M) * H * 2);
  DA(p->q, static_cast<size_t>(M) * QD * 2);
  const int NTlm = p->full ? p->V / 128 : 0;
  if (p->full) {
    DA(p->hfin, static_cast<size_t>(Mr) * H * 2);
    DA(p->rfin, static_cast<size_t>(M) * H * 2);
    DA(p->logits, static_cast<size_t>(M) * p->V * 4);
    DA(p->best_val, static_cast<size_t>(NTlm) * M * 4);
    DA(p->best_idx, static_cast<size_t>(NTlm) * M * 4);
  }
  // RoPE table [max_context][d/2] (cos, sin), computed in double
  {
    const int maxp = c.max_context, half = p->d / 2;
    std::vector<float> tab(static_cast<size_t>(maxp) * half * 2);
    for (int pos = 0; pos < maxp; ++pos)
      for (int i = 0; i < half; ++i) {
        const double inv = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / p->d);
        const double ang = static_cast<double>(pos) * inv;
        tab[(static_cast<size_t>(pos) * half + i) * 2] = static_cast<float>(std::cos(ang));
        tab[(static_cast<size_t>(pos) * half + i) * 2 + 1] = static_cast<float>(std::sin(ang));
      }
    DA(p->rope, tab.size() * 4);
    CK(cudaMemcpy(p->rope, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice));
  }
  // workspaces: partial sums of the widest GEMM / attention split
  {
    const int npair = 2;
    const size_t gws = static_cast<size_t>(p->sms) * 2 * npair * p->Mp * 128 * 4;
    DA(p->ws_gemm[0], gws);
    DA(p->ws_gemm[1], gws);
    const int QR = p->T * (p->Hq / p->Hkv);
    const int QRp = QR <= 16 ? 16 : (QR <= 32 ? 32 : 64);
    DA(p->ws_attn, static_cast<size_t>(p->sms) * 2 * QRp * 129 * 4);
  }
  // tensor maps: 4 per layer (weights), 4 activations, lm_head + its input
  const int n_maps = 4 * p->L + 4 + (p->full ? 2 : 0);
  p->h_maps.resize(n_maps);
  {
    void* m = nullptr;
    if ((s = dev_alloc(p, &m, sizeof(CUtensorMap) * n_maps)) != DL_OK) return s;
    p->d_maps = static_cast<CUtensorMap*>(m);
  }
  const uint32_t xrows = static_cast<uint32_t>(p->mma ? p->Mp : p->M);
  auto wmap = [&](int idx, const void* w, int N, int K) -> bool {
    if (!w || !aligned16(w)) return false;
    return encode_map(&p->h_maps[idx], w, p->fp8, K, N, 128);
  };
  for (int l = 0; l < p->L; ++l) {
    const dl_layer_weights& lw = p->layers[l];
    if (!lw.ln1_w || !lw.ln2_w || !lw.q_norm_w || !lw.k_norm_w)
      return fail(DL_ERR_INVALID_ARG, "norm weight pointer is NULL");
    if (p->fp8 && (!lw.w_qkv_scale || !lw.w_o_scale || !lw.w_gate_up_scale || !lw.w_down_scale))
      return fail(DL_ERR_INVALID_ARG, "FP8 weights need scale pointers");
    if (!wmap(4 * l + 0, lw.w_qkv, (p->Hq + 2 * p->Hkv) * p->d, H) ||
        !wmap(4 * l + 1, lw.w_o, H, QD) || !wmap(4 * l + 2, lw.w_gate_up, 2 * I, H) ||
        !wmap(4 * l + 3, lw.w_down, H, I))
      return fail(DL_ERR_INVALID_ARG, "weight pointer NULL, unaligned or not encodable");
  }
  const int xm = 4 * p->L;
  if (!encode_map(&p->h_maps[xm + 0], p->h1, p->fp8, H, xrows, xrows) ||
      !encode_map(&p->h_maps[xm + 1], p->attn, p->fp8, QD, xrows, xrows) ||
      !encode_map(&p->h_maps[xm + 2], p->h2, p->fp8, H, xrows, xrows) ||
      !encode_map(&p->h_maps[xm + 3], p->act, p->fp8, I, xrows, xrows))
    return fail(DL_ERR_CUDA, "activation tensor map encode failed");
  if (p->full) {
    if (!c.lm_head_w || !aligned16(c.lm_head_w) || !c.final_norm_w)
      return fail(DL_ERR_INVALID_ARG, "lm_head / final norm pointer invalid");
    if (!encode_map(&p->h_maps[xm + 4], c.lm_head_w, false, H, p->V, 128) ||
        !encode_map(&p->h_maps[xm + 5], p->hfin, false, H, xrows, xrows))
      return fail(DL_ERR_CUDA, "lm_head tensor map encode failed");
  }
  CK(cudaMemcpy(p->d_maps, p->h_maps.data(), sizeof(CUtensorMap) * n_maps,
                cudaMemcpyHostToDevice));

  // counters: per op its own slice (tile / pair counters + one done counter)
  const int ntq = p->Hq + 2 * p->Hkv;
  const size_t per_layer = (ntq + 1) * 2 + (p->R * p->Hkv + 1) + (H / 128 + 1) + (I / 128 + 1) +
                           (H / 128 + 1) + 8;
  p->n_counters = per_layer * p->L + (NTlm + 1) + 16;
  DA(p->counters, p->n_counters * sizeof(unsigned));
  size_t cpos = 0;
  auto take = [&](size_t n) {
    unsigned* r = p->counters + cpos;
    cpos += n;
    return r;
  };

  const size_t MH2 = static_cast<size_t>(M) * H * 2;
  if (const char* e = std::getenv("DL_ATTN")) p->attn_tc = std::strcmp(e, "mma_sync") != 0;
  if (const char* e = std::getenv("DL_MEGA_HEAD_EVENTS")) p->head_events = std::atoi(e) != 0;
  if (const char* e = std::getenv("DL_DEFER_FIXUP")) p->defer_fixup = std::atoi(e) != 0;
  if (const char* e = std::getenv("DL_ATTN_KV4")) p->attn_kv4 = std::atoi(e) != 0;
  if (const char* e = std::getenv("DL_ATTN_MIN_BLOCKS")) p->attn_min_blocks = std::max(1, std::atoi(e));
  if (const char* e = std::getenv("DL_ATTN_PRE_STAGES")) p->attn_pre_stages = std::max(0, std::atoi(e));
  if (const char* e = std::getenv("DL_NORM_SPLIT")) p->norm_split = std::max(1, std::min(4, std::atoi(e)));
  if (const char* e = std::getenv("DL_ATTN_SPLIT_SOFTMAX")) p->split_sm = std::atoi(e) != 0;
  if (const char* e = std::getenv("DL_DAG_PROGRAMMATIC_EDGES")) p->dag_prog_edges = std::atoi(e) != 0;
  if (const char* e = std::getenv("DL_GEMM_STAGES")) p->gemm_stages_max = std::max(2, std::min(kMaxStages, std::atoi(e)));
  if (const char* e = std::getenv("DL_ATTN_STAGES")) p->attn_stages_max = std::max(2, std::min(kMaxStages, std::atoi(e)));
  for (int l = 0; l < p->L; ++l) {
    const dl_layer_weights& lw = p->layers[l];
    const bool last = (l == p->L - 1);
    const CUtensorMap* tm = p->d_maps;
    // 1. residual add + RMSNorm (+ quant)
    LaunchOp n1 = make_norm(p, l == 0 ? bound(SLOT_X) : fixed(p->y),
                            l == 0 ? bound(SLOT_RES) : fixed(p->r2), fixed(p->r1), lw.ln1_w, p->h1,
                            p->h1s, p->fp8, "add_rmsnorm1");
    // 2. QKV projection + QK-norm + RoPE + paged KV write
    GemmSpec qs{tm + 4 * l + 0, tm + xm + 0, lw.w_qkv_scale, p->h1s, p->fp8, H, ntq, 0, false, 0,
                EPI_QKV_ROPE, 0, "qkv_rope_kvwrite"};
    auto fill_qkv = [&](LaunchOp& op) {
      GemmArgs& a = op.args.gemm;
      a.q_out = p->q;
      a.kv = bound(SLOT_KV);
      a.bt = bound(SLOT_BT);
      a.pos = bound(SLOT_POS);
      a.q_norm_w = lw.q_norm_w;
      a.k_norm_w = lw.k_norm_w;
      a.rope_cs = p->rope;
      a.rope_max_pos = c.max_context;
      a.Hq = p->Hq;
      a.Hkv = p->Hkv;
      a.d = p->d;
      a.T = p->T;
      a.P = p->P;
      a.num_pages = c.num_pages;
      a.max_pages = c.max_pages_per_request;
      a.layer = l;
      a.eps = c.eps;
    };
    LaunchOp qkv = make_gemm(p, qs, take(ntq + 1));
    fill_qkv(qkv);
    // DAG variant: q heads on the main chain, k/v heads on a side branch
    GemmSpec qq = qs;
    qq.NT = p->Hq;
    qq.name = "q_rope";
    LaunchOp qop = make_gemm(p, qq, take(p->Hq + 1));
    fill_qkv(qop);
    GemmSpec qkvs = qs;
    qkvs.NT = 2 * p->Hkv;
    qkvs.t_base = p->Hq;
    qkvs.ws_slot = 1;
    qkvs.name = "kv_rope_write";
    LaunchOp kvop = make_gemm(p, qkvs, take(2 * p->Hkv + 1));
    fill_qkv(kvop);
    kvop.branch = 1;
    // 3. attention
    LaunchOp at = make_attn(p, l, take(p->R * p->Hkv + 1));
    // 4. O projection
    GemmSpec os{tm + 4 * l + 1, tm + xm + 1, lw.w_o_scale, p->attns, p->fp8, QD, H / 128, 0,
                false, 0, EPI_STORE_BF16, 0, "o_proj"};
    LaunchOp oop = make_gemm(p, os, take(H / 128 + 1));
    oop.args.gemm.out = fixed(p->o2);
    oop.args.gemm.ldo = H;
    // 5. residual add + RMSNorm (+ quant)
    const DPtr r2dst = (last && !p->full) ? bound(SLOT_OUT, static_cast<long long>(MH2)) : fixed(p->r2);
    LaunchOp n2 = make_norm(p, fixed(p->o2), fixed(p->r1), r2dst, lw.ln2_w, p->h2, p->h2s, p->fp8,
                            "add_rmsnorm2");
    // 6. gate/up + SiLU*mul (+ quant)
    GemmSpec gs{tm + 4 * l + 2, tm + xm + 2, lw.w_gate_up_scale, p->h2s, p->fp8, H, I / 128, 0,
                true, I, EPI_SILU_MUL, 0, "gate_up_silu"};
    LaunchOp gop = make_gemm(p, gs, take(I / 128 + 1));
    gop.args.gemm.act = p->act;
    gop.args.gemm.act_scale = p->acts;
    gop.args.gemm.act_ld = I;
    // 7. down projection
    GemmSpec ds{tm + 4 * l + 3, tm + xm + 3, lw.w_down_scale, p->acts, p->fp8, I, H / 128, 0,
                false, 0, EPI_STORE_BF16, 0, "down_proj"};
    LaunchOp dop = make_gemm(p, ds, take(H / 128 + 1));
    dop.args.gemm.out = (last && !p->full) ? bound(SLOT_OUT, 0) : fixed(p->y);
    dop.args.gemm.ldo = H;

    for (LaunchOp* op : {&n1, &qkv, &at, &oop, &n2, &gop, &dop}) p->lin.push_back(*op);
    LaunchOp at_join = at;
    at_join.branch = 2;
    for (LaunchOp* op : {&n1, &qop, &kvop, &at_join, &oop, &n2, &gop, &dop}) p->dag.push_back(*op);
  }
  if (p->full) {
    LaunchOp nf = make_norm(p, fixed(p->y), fixed(p->r2), fixed(p->rfin), c.final_norm_w, p->hfin,
                            nullptr, false, "final_norm");
    const CUtensorMap* tm = p->d_maps;
    GemmSpec ls{tm + xm + 4, tm + xm + 5, nullptr, nullptr, false, H, NTlm, 0, false, 0, EPI_LOGITS,
                0, "lm_head_argmax"};
    LaunchOp lop = make_gemm(p, ls, take(NTlm + 1));
    lop.args.gemm.out = fixed(p->logits);
    lop.args.gemm.ldo = p->V;
    lop.args.gemm.best_val = p->best_val;
    lop.args.gemm.best_idx = p->best_idx;
    lop.args.gemm.ids = bound(SLOT_OUT);
    p->lin.push_back(nf);
    p->lin.push_back(lop);
    p->dag.push_back(nf);
    p->dag.push_back(lop);
  }
  if (cpos > p->n_counters) return fail(DL_ERR_CUDA, "counter pool overflow");
  if (p->defer_fixup)
    for (auto* list : {&p->lin, &p->dag}) defer_fixups(*list);

  // the kernels split units with 32-bit arithmetic: units x CTAs < 2^32
  for (const auto* list : {&p->lin, &p->dag})
    for (const LaunchOp& op : *list) {
      long long U = 0, G = 1;
      if (op.args.kind == OP_GEMM) {
        U = static_cast<long long>(op.args.gemm.NT) * op.args.gemm.KB;
        G = op.args.gemm.G;
      } else if (op.args.kind == OP_ATTN) {
        U = static_cast<long long>(op.args.attn.R) * op.args.attn.Hkv * op.args.attn.NB;
        G = op.args.attn.G;
      }
      if (U * G >= (1LL << 32)) return fail(DL_ERR_PLAN_INVALID, "too many work units for one op");
    }
  if (const char* e = std::getenv("DL_L2_PREFETCH_UNITS")) p->pf_units = std::atoi(e);
  // L2 prefetch: an attention or a projection directly followed (on the
  // same stream) by a projection warms L2 with the weight tiles that
  // projection's first stages load, once its own loads are out
  for (auto* list : {&p->lin, &p->dag})
    for (size_t i = 0; i + 1 < list->size(); ++i) {
      LaunchOp& cur = (*list)[i];
      const LaunchOp& nx = (*list)[i + 1];
      if (nx.args.kind != OP_GEMM || nx.branch != 0 || cur.branch != 0) continue;
      // not from a norm: its M CTAs (one at batch 1) would issue the whole
      // projection's prefetches through their own TMA units (measured: 38
      // and 78 us before the QKV and gate/up projections at batch 1), and
      // under programmatic dependent launch the projection's CTAs load their
      // first stages during the norm themselves
      if (cur.args.kind == OP_NORM) continue;
      const GemmArgs& g = nx.args.gemm;
      PrefetchSpec pf;
      pf.tmap = g.tmap_w;
      pf.NT = g.NT;
      pf.KB = g.KB;
      pf.G = g.G;
      pf.t_base = g.t_base;
      pf.pair = g.pair;
      pf.up_row = g.up_row;
      pf.kel = 128 / (g.fp8 ? 1 : 2);
      // 4 units (64 KiB, or 128 KiB of gate + up) per share measured best:
      // enough to cover the hand-over, little enough not to queue ahead of
      // the boundary's own latency-bound reads
      pf.units = std::max(0, p->pf_units);
      if (pf.units == 0) pf.tmap = nullptr;
      if (cur.args.kind == OP_ATTN) cur.args.attn.pf = pf;
      else if (cur.args.kind == OP_GEMM) cur.args.gemm.pf = pf;
    }

  // kernel attributes: dynamic shared memory (the largest user of each kernel)
  int max_smem = 0;
  {
    std::vector<std::pair<const void*, int>> need;
    for (const auto* list : {&p->lin, &p->dag})
      for (const LaunchOp& op : *list) {
        bool found = false;
        for (auto& kv : need)
          if (kv.first == op.kernel) {
            kv.second = std::max(kv.second, op.smem);
            found = true;
          }
        if (!found) need.emplace_back(op.kernel, op.smem);
        max_smem = std::max(max_smem, op.smem);
      }
    for (auto& kv : need)
      CK(cudaFuncSetAttribute(kv.first, cudaFuncAttributeMaxDynamicSharedMemorySize, kv.second));
  }

  // streams / events for capture and the DAG fork
  CK(cudaStreamCreateWithFlags(&p->cap, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking));
  CK(cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming));
  CK(cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming));

  // trace build (DL_TRACE=1 in the environment at creation)
  {
    const char* tr = std::getenv("DL_TRACE");
    if (tr && tr[0] == '1' && tr[1] == 0) {
      p->trace_ops = static_cast<int>(std::max(p->lin.size(), p->dag.size()));
      DA(p->d_trace, static_cast<size_t>(p->trace_ops) * p->sms * kTraceSlots * 8);
    }
  }

  // e2e staging buffers
  DA(p->st_x, MH2);
  DA(p->st_res, MH2);
  DA(p->st_bt, static_cast<size_t>(p->R) * c.max_pages_per_request * 4);
  DA(p->st_pos, static_cast<size_t>(M) * 4);
  DA(p->st_out, p->full ? static_cast<size_t>(M) * 4 : 2 * MH2);

  // megakernel
  if (c.modes_mask & (1u << DL_MODE_MEGAKERNEL)) {
    p->mega = p->lin;
    for (LaunchOp& op : p->mega) {
      if (op.args.kind == OP_GEMM && op.args.gemm.epi == EPI_PARTIALS) op.args.gemm.epi = EPI_STORE_BF16;
      if (op.args.kind == OP_NORM) op.args.norm.part = nullptr;   // (split rows: see NormArgs)
    }
    if ((s = build_mega(p)) != DL_OK) return s;
    if ((s = validate_mega(p)) != DL_OK) return s;
    // the worker's ring of equal operand slots (32 KiB of weight tiles or
    // K/V plus the activation slices) and the largest private area
    int slot = 32768, priv = norm_smem_bytes();
    for (const LaunchOp& op : p->mega) {
      if (op.args.kind == OP_GEMM) {
        const GemmArgs& a = op.args.gemm;
        slot = std::max(slot, 32768 + (a.pair ? 1 : 2) * (((a.Mp * 128 + 1023) / 1024) * 1024));
        priv = std::max(priv, gemm_smem_bytes(a.pair ? 2 : 1, a.Mp, 0, a.KB, a.fp8, a.epi, a.M,
                                              a.share_max));
      } else if (op.args.kind == OP_ATTN) {
        priv = std::max(priv, attn_smem_bytes(op.args.attn.QRp, 0));
      }
    }
    priv = (priv + 1023) & ~1023;
    cudaFuncAttributes fa;
    CK(cudaFuncGetAttributes(&fa, mega_kernel()));
    int optin = 0;
    CK(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->dev));
    const int avail = optin - static_cast<int>(fa.sharedSizeBytes) - 1024 - priv;
    p->mega_ns = std::min(kMaxSlots, avail / slot);
    // two slots suffice for progress (the producer issues every pending
    // activation slice before it waits for a slot); fewer cannot hold a unit
    // while the next one streams in
    if (p->mega_ns < 2) return fail(DL_ERR_PLAN_INVALID, "megakernel ring has fewer than 2 slots");
    p->mega_slot = slot;
    p->mega_priv_off = p->mega_ns * slot;
    p->mega_smem = 1024 + p->mega_priv_off + priv;
    (void)max_smem;
    CK(cudaFuncSetAttribute(mega_kernel(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                            p->mega_smem));
    int per_sm = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mega_kernel(), kThreads,
                                                     p->mega_smem));
    if (per_sm < 1) return fail(DL_ERR_PLAN_INVALID, "megakernel worker does not fit on an SM");
    std::vector<OpArgs> h_ops;
    for (const LaunchOp& op : p->mega) h_ops.push_back(op.args);
    DA(p->d_ops, h_ops.size() * sizeof(OpArgs));
    CK(cudaMemcpy(p->d_ops, h_ops.data(), h_ops.size() * sizeof(OpArgs), cudaMemcpyHostToDevice));
    DA(p->d_queues, p->queues.size() * sizeof(Instr));
    if ((s = upload_mega(p)) != DL_OK) return s;
    DA(p->d_events, static_cast<size_t>(p->n_events) * 4);
    DA(p->d_finish, 64);
  }
#undef DA
  CK(cudaDeviceSynchronize());
  // graphs
  for (int mode : {DL_MODE_PDL_GRAPH, DL_MODE_GRAPH_LINEAR, DL_MODE_GRAPH_LINEAR_PDL,
                   DL_MODE_GRAPH_DAG})
    if (c.modes_mask & (1u << mode))
      if ((s = capture_graph(p, mode)) != DL_OK) return s;
  return DL_OK;
}

extern "C" dl_plan* dl_plan_create(const dl_config* cfg) {
  if (check_config(cfg) != DL_OK) return nullptr;
  dl_plan* p = new dl_plan();
  p->cfg = *cfg;
  p->layers.assign(cfg->layers, cfg->layers + cfg->n_layers);
  p->cfg.layers = nullptr;
  const dl_status s = build_plan(p);
  if (s != DL_OK) {
    const std::string msg = g_err;
    free_plan(p);
    g_err = msg;
    return nullptr;
  }
  g_err.clear();
  return p;
}

extern "C" void dl_plan_destroy(dl_plan* p) {
  if (p) cudaDeviceSynchronize();
  free_plan(p);
}

// ------------------------------------------------------------------ steps
static dl_status bind(dl_plan* p, Binding& b, cudaStream_t s) {
  if (p->have_last && std::memcmp(b.p, p->last.p, sizeof(b.p)) == 0) return DL_OK;
  // TMA descriptor of the bound cache, [rows, head_dim] bf16
  const uint64_t rows = static_cast<uint64_t>(p->L) * p->cfg.num_pages * 2 * p->Hkv * p->P;
  const uint32_t box = static_cast<uint32_t>(std::min(p->P, kAttnKeys));
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(p->d), rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(p->d) * 2};
  cuuint32_t boxd[2] = {64, box};
  cuuint32_t estr[2] = {1, 1};
  if (g_encode(&b.kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, b.p[SLOT_KV], dims, strides, boxd,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return fail(DL_ERR_INVALID_ARG, "kv_pages cannot be described by a TMA descriptor");
  if (p->attn_tc && p->attn_kv4 && p->P % kAttnKeys == 0 && p->d == 128) {
    // [K/V][d-half][rows][64 elements]: strides one row, 128 bytes, and
    // kv_heads * page_size rows (V of a slot lies that far after its K)
    const uint64_t row_b = static_cast<uint64_t>(p->d) * 2;
    cuuint64_t dims4[4] = {64, rows, 2, 2};
    cuuint64_t strides4[3] = {row_b, 128, static_cast<cuuint64_t>(p->Hkv) * p->P * row_b};
    cuuint32_t boxd4[4] = {64, static_cast<cuuint32_t>(kAttnKeys), 2, 2};
    cuuint32_t estr4[4] = {1, 1, 1, 1};
    if (g_encode(&b.kv_map4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, b.p[SLOT_KV], dims4, strides4,
                 boxd4, estr4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return fail(DL_ERR_INVALID_ARG, "kv_pages cannot be described by a 4-D TMA descriptor");
  }
  CK(launch_bind(p->d_binding, b, s));
  p->last = b;
  p->have_last = true;
  return DL_OK;
}

extern "C" dl_status dl_decode_step(dl_plan* p, const void* x, const void* residual,
                                    void* kv_pages, const int32_t* block_table,
                                    const int32_t* positions, void* out, int mode, void* stream) {
  if (!p) return fail(DL_ERR_INVALID_ARG, "plan is NULL");
  if (!x || !residual || !kv_pages || !block_table || !positions || !out)
    return fail(DL_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(x) || !aligned16(residual) || !aligned16(kv_pages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3) || (reinterpret_cast<uintptr_t>(positions) & 3))
    return fail(DL_ERR_INVALID_ARG, "misaligned tensor pointer");
  if (mode < 0 || mode > 5) return fail(DL_ERR_INVALID_ARG, "unknown mode");
  if (mode != DL_MODE_SERIAL && !(p->cfg.modes_mask & (1u << mode)))
    return fail(DL_ERR_INVALID_ARG, "mode not prepared (modes_mask)");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Binding b;
  std::memset(&b, 0, sizeof(b));
  b.p[SLOT_X] = const_cast<void*>(x);
  b.p[SLOT_RES] = const_cast<void*>(residual);
  b.p[SLOT_KV] = kv_pages;
  b.p[SLOT_BT] = const_cast<int32_t*>(block_table);
  b.p[SLOT_POS] = const_cast<int32_t*>(positions);
  b.p[SLOT_OUT] = out;
  dl_status st = bind(p, b, s);
  if (st != DL_OK) return st;
  switch (mode) {
    case DL_MODE_SERIAL: {
      for (size_t i = 0; i < p->lin.size(); ++i) CK(launch_op(p, p->lin[i], s, false, static_cast<int>(i)));
      break;
    }
    case DL_MODE_MEGAKERNEL:
      CK(launch_mega(p, s));
      break;
    default:
      CK(cudaGraphLaunch(p->exec[mode], s));
      break;
  }
  return DL_OK;
}

extern "C" dl_status dl_decode_step_host(dl_plan* p, const void* x_host, const void* residual_host,
                                         void* kv_pages, const int32_t* block_table_host,
                                         const int32_t* positions_host, void* out_host, int mode,
                                         void* stream) {
  if (!p) return fail(DL_ERR_INVALID_ARG, "plan is NULL");
  if (!x_host || !residual_host || !block_table_host || !positions_host || !out_host)
    return fail(DL_ERR_INVALID_ARG, "NULL host pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t MH2 = static_cast<size_t>(p->M) * p->H * 2;
  // Host buffers the device can address (page-locked and mapped: every
  // page-locked allocation under unified addressing) are used in place: the
  // first kernels read the inputs across the host link and the last ones
  // write the result there, with no copy of its own on the stream (each
  // copy costs a few microseconds of latency however small it is).  Any
  // other buffer goes through the plan's staging copies.
  auto device_view = [](const void* h) -> void* {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
      cudaGetLastError();   // not a CUDA-known pointer: clear the error
      return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
    return (reinterpret_cast<uintptr_t>(at.devicePointer) & 15) == 0 ? at.devicePointer : nullptr;
  };
  void* dx = device_view(x_host);
  void* dres = device_view(residual_host);
  void* dbt = device_view(block_table_host);
  void* dpos = device_view(positions_host);
  void* dout = device_view(out_host);
  if (dx && dres && dbt && dpos && dout)
    return dl_decode_step(p, dx, dres, kv_pages, static_cast<const int32_t*>(dbt),
                          static_cast<const int32_t*>(dpos), dout, mode, stream);
  CK(cudaMemcpyAsync(p->st_x, x_host, MH2, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(p->st_res, residual_host, MH2, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(p->st_bt, block_table_host,
                     static_cast<size_t>(p->R) * p->cfg.max_pages_per_request * 4,
                     cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(p->st_pos, positions_host, static_cast<size_t>(p->M) * 4,
                     cudaMemcpyHostToDevice, s));
  const dl_status st = dl_decode_step(p, p->st_x, p->st_res, kv_pages, p->st_bt, p->st_pos,
                                      p->st_out, mode, stream);
  if (st != DL_OK) return st;
  CK(cudaMemcpyAsync(out_host, p->st_out, p->full ? static_cast<size_t>(p->M) * 4 : 2 * MH2,
                     cudaMemcpyDeviceToHost, s));
  return DL_OK;
}

extern "C" dl_status dl_plan_status(dl_plan* p) {
  if (!p) return fail(DL_ERR_INVALID_ARG, "plan is NULL");
  DevStatus st;
  CK(cudaMemcpy(&st, p->d_status, sizeof(st), cudaMemcpyDeviceToHost));
  if (st.code == DERR_NONE) return DL_OK;
  char buf[256];
  std::snprintf(buf, sizeof(buf), "device error %u: op %u cta %u where %u value %u (block %u thread %u)",
                st.code, st.info[0], st.info[1], st.info[2], st.info[3], st.info[4], st.info[5]);
  // clear the status and every counter a failed step may have left raised
  CK(cudaMemset(p->d_status, 0, sizeof(DevStatus)));
  CK(cudaMemset(p->counters, 0, p->n_counters * sizeof(unsigned)));
  if (p->d_events) CK(cudaMemset(p->d_events, 0, static_cast<size_t>(p->n_events) * 4));
  if (p->d_finish) CK(cudaMemset(p->d_finish, 0, 64));
  CK(cudaDeviceSynchronize());
  return fail(st.code == DERR_TIMEOUT ? DL_ERR_TIMEOUT
              : st.code == DERR_BOUNDS ? DL_ERR_DEVICE_BOUNDS
                                       : DL_ERR_CUDA,
              buf);
}

extern "C" const float* dl_plan_logits(dl_plan* p) { return p ? p->logits : nullptr; }

extern "C" dl_status dl_plan_trace(dl_plan* p, void* host_buf, size_t bytes, int* n_ops,
                                   int* n_ctas) {
  if (!p) return fail(DL_ERR_INVALID_ARG, "plan is NULL");
  if (!p->d_trace) return fail(DL_ERR_UNSUPPORTED, "plan was created without DL_TRACE=1");
  if (n_ops) *n_ops = p->trace_ops;
  if (n_ctas) *n_ctas = p->sms;
  if (!host_buf) return DL_OK;
  const size_t need = static_cast<size_t>(p->trace_ops) * p->sms * kTraceSlots * 8;
  if (bytes < need) return fail(DL_ERR_INVALID_ARG, "trace buffer too small");
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(host_buf, p->d_trace, need, cudaMemcpyDeviceToHost));
  CK(cudaMemset(p->d_trace, 0, need));
  CK(cudaDeviceSynchronize());
  return DL_OK;
}

extern "C" dl_status dl_plan_debug_buffer(dl_plan* p, int which, void** ptr, size_t* bytes) {
  if (!p || !ptr || !bytes) return fail(DL_ERR_INVALID_ARG, "NULL argument");
  const size_t eb = p->fp8 ? 1 : 2, M = p->M, Mr = p->Mrows, H = p->H, I = p->I;
  const size_t QD = static_cast<size_t>(p->Hq) * p->d;
  switch (which) {
    case 0: *ptr = p->r1; *bytes = M * H * 2; break;
    case 1: *ptr = p->h1; *bytes = Mr * H * eb; break;
    case 2: *ptr = p->h1s; *bytes = M * (H / 128) * 4; break;
    case 3: *ptr = p->q; *bytes = M * QD * 2; break;
    case 4: *ptr = p->attn; *bytes = Mr * QD * eb; break;
    case 5: *ptr = p->attns; *bytes = M * (QD / 128) * 4; break;
    case 6: *ptr = p->o2; *bytes = M * H * 2; break;
    case 7: *ptr = p->r2; *bytes = M * H * 2; break;
    case 8: *ptr = p->h2; *bytes = Mr * H * eb; break;
    case 9: *ptr = p->h2s; *bytes = M * (H / 128) * 4; break;
    case 10: *ptr = p->act; *bytes = Mr * I * eb; break;
    case 11: *ptr = p->acts; *bytes = M * (I / 128) * 4; break;
    case 12: *ptr = p->y; *bytes = M * H * 2; break;
    case 16:
      if (!p->full) return fail(DL_ERR_INVALID_ARG, "debug buffer 16 (final norm) needs a full-step plan");
      *ptr = p->hfin;
      *bytes = M * H * 2;
      break;
    default: return fail(DL_ERR_INVALID_ARG, "unknown debug buffer");
  }
  return DL_OK;
}

extern "C" int dl_plan_kernel_count(dl_plan* p, int mode) {
  if (!p) return -1;
  if (mode == DL_MODE_MEGAKERNEL) return 1;
  if (mode == DL_MODE_PDL_GRAPH || mode == DL_MODE_GRAPH_DAG) return static_cast<int>(p->dag.size());
  return static_cast<int>(p->lin.size());
}

extern "C" int dl_plan_op_count(dl_plan* p) { return p ? static_cast<int>(p->lin.size()) : -1; }

extern "C" dl_status dl_plan_op_info(dl_plan* p, int i, char* name, size_t name_len, int* grid,
                                     int* smem_bytes) {
  if (!p || i < 0 || i >= static_cast<int>(p->lin.size()))
    return fail(DL_ERR_INVALID_ARG, "op index out of range");
  const LaunchOp& op = p->lin[i];
  if (name && name_len) {
    std::strncpy(name, op.name.c_str(), name_len - 1);
    name[name_len - 1] = 0;
  }
  if (grid) *grid = op.grid;
  if (smem_bytes) *smem_bytes = op.smem;
  return DL_OK;
}

extern "C" dl_status dl_plan_launch_op(dl_plan* p, int i, void* stream) {
  if (!p || i < 0 || i >= static_cast<int>(p->lin.size()))
    return fail(DL_ERR_INVALID_ARG, "op index out of range");
  if (!p->have_last) return fail(DL_ERR_INVALID_ARG, "no operands bound yet");
  CK(launch_op(p, p->lin[i], static_cast<cudaStream_t>(stream), false, i));
  return DL_OK;
}

extern "C" dl_status dl_plan_launch_ops(dl_plan* p, int first, int count, int pdl,
                                        int gdc_mode, void* stream) {
  if (!p || first < 0 || count < 1 || first + count > static_cast<int>(p->lin.size()))
    return fail(DL_ERR_INVALID_ARG, "op range out of range");
  if (gdc_mode < 0 || gdc_mode > 2) return fail(DL_ERR_INVALID_ARG, "gdc_mode must be 0, 1 or 2");
  if (!p->have_last) return fail(DL_ERR_INVALID_ARG, "no operands bound yet");
  for (int i = first; i < first + count; ++i) {
    LaunchOp op = p->lin[i];
    if (op.args.kind == OP_GEMM) op.args.gemm.gdc_mode = gdc_mode;
    CK(launch_op(p, op, static_cast<cudaStream_t>(stream), pdl != 0, i));
  }
  return DL_OK;
}

extern "C" dl_status dl_plan_mega_info(dl_plan* p, int* workers, int* qlen, int* events) {
  if (!p || !p->d_queues) return fail(DL_ERR_INVALID_ARG, "no megakernel plan");
  if (workers) *workers = p->workers;
  if (qlen) *qlen = p->qlen;
  if (events) *events = p->n_events;
  return DL_OK;
}

// Test-only: the megakernel queue validator on a host array of
// instructions (the layout of include/dl.h's dl_test_validate_mega_queues).
extern "C" dl_status dl_test_validate_mega_queues(const void* queues, int workers, int qlen,
                                                  int n_events) {
  if (!queues || workers <= 0 || qlen <= 0 || n_events <= 0)
    return fail(DL_ERR_INVALID_ARG, "empty queue description");
  return validate_queues(static_cast<const Instr*>(queues), workers, qlen, n_events);
}

extern "C" dl_status dl_plan_debug_perturb_wait(dl_plan* p, unsigned delta,
                                                unsigned long long budget_ns, int validate) {
  if (!p || !p->d_queues) return fail(DL_ERR_INVALID_ARG, "no megakernel plan");
  static const unsigned long long kDefault = 1000000000ull;
  // worker 0's first instruction with a wait
  if (p->perturb_idx < 0) {
    for (int i = 0; i < p->qlen; ++i) {
      const Instr& in = p->queues[i];
      if (in.op_row != 0xffffffffu && in.n_wait > 0) {
        p->perturb_idx = i;
        p->perturb_orig = in.wait_value[0];
        break;
      }
    }
  }
  if (p->perturb_idx < 0) return fail(DL_ERR_INVALID_ARG, "no waiting instruction");
  Instr* target = &p->queues[p->perturb_idx];
  const unsigned base_value = p->perturb_orig;
  target->wait_value[0] = base_value + delta;
  p->budget_ns = delta ? budget_ns : kDefault;
  if (validate) {
    const dl_status v = validate_mega(p);
    if (v != DL_OK) {
      target->wait_value[0] = base_value;
      p->budget_ns = kDefault;
      return v;
    }
  }
  return upload_mega(p);
}

// ------------------------------------------------------------ test hooks
extern "C" dl_status dl_test_kv_write(const void* src, void* kv_pages, const int32_t* block_table,
                                      const int32_t* positions, int layer, int M, int T,
                                      int n_kv_heads, int head_dim, int page_size, int num_pages,
                                      int max_pages, void* stream) {
  if (!src || !kv_pages || !block_table || !positions || M <= 0 || T <= 0)
    return fail(DL_ERR_INVALID_ARG, "bad argument");
  static DevStatus* st = nullptr;
  if (!st && cudaMalloc(&st, sizeof(DevStatus)) == cudaSuccess) cudaMemset(st, 0, sizeof(DevStatus));
  CK(launch_test_kv_write(src, kv_pages, block_table, positions, layer, M, T, n_kv_heads, head_dim,
                          page_size, num_pages, max_pages, st, static_cast<cudaStream_t>(stream)));
  return DL_OK;
}

extern "C" dl_status dl_test_kv_gather(const void* kv_pages, const int32_t* block_table, void* dst,
                                       int layer, int R, int n_keys, int n_kv_heads, int head_dim,
                                       int page_size, int num_pages, int max_pages, void* stream) {
  if (!kv_pages || !block_table || !dst || R <= 0 || n_keys <= 0)
    return fail(DL_ERR_INVALID_ARG, "bad argument");
  static DevStatus* st = nullptr;
  if (!st && cudaMalloc(&st, sizeof(DevStatus)) == cudaSuccess) cudaMemset(st, 0, sizeof(DevStatus));
  CK(launch_test_kv_gather(kv_pages, block_table, dst, layer, R, n_keys, n_kv_heads, head_dim,
                           page_size, num_pages, max_pages, st, static_cast<cudaStream_t>(stream)));
  return DL_OK;
}
