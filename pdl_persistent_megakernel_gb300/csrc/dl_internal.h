// dl_internal.h -- structures shared by the host planner and the device code
// of the decode-step library (not part of the public C ABI).
//
// Every operation of the decode step is a "tile engine" that a CTA runs over
// its share of the operation's work.  The same engine runs inside the
// standalone kernels (serial and graph schedules, one kernel per operation)
// and inside the persistent megakernel (one instruction per CTA share), so
// the three schedules differ only in how shares are ordered on the GPU.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda.h>

namespace dl {

// ------------------------------------------------------------------ limits
constexpr int kThreads = 288;        // 9 warps: warp 0 loads, warps 1-8 compute
constexpr int kConsumerThreads = 256;
constexpr int kBN = 128;             // weight rows per GEMM tile
constexpr int kBKBytes = 128;        // bytes of K per pipeline stage (one
                                     // 128-byte swizzle atom: 64 bf16 / 128 e4m3)
constexpr int kMaxM = 64;            // tokens per step
constexpr int kAttnKeys = 64;        // keys per attention pipeline stage
constexpr int kMaxQRows = 64;        // query rows per (request, kv head)
constexpr int kMaxStages = 12;
constexpr int kMaxSlots = 16;        // operand slots of a megakernel worker's ring

// ----------------------------------------------------- runtime bindings
// Pointers supplied per decode call (the caller's tensors).  Kernels read
// them from a small device table so that captured graphs and megakernel
// queues stay valid when the caller passes new buffers.
enum BindingSlot : int {
  SLOT_X = 0,        // bf16 [M, H]          layer-0 input
  SLOT_RES = 1,      // bf16 [M, H]          layer-0 residual
  SLOT_KV = 2,       // bf16 paged KV cache [L][pages][2][Hkv][P][d]
  SLOT_BT = 3,       // int32 [R, max_pages] block table
  SLOT_POS = 4,      // int32 [M]            positions
  SLOT_OUT = 5,      // bf16 [2, M, H] (layer plans) / int32 [M] (full plans)
  NUM_SLOTS = 8
};

struct alignas(128) Binding {
  void* p[NUM_SLOTS];
  // TMA descriptor of the bound KV cache viewed as [rows, head_dim] bf16
  // (rows = layers * pages * 2 * kv_heads * page_size), 128-byte swizzle,
  // boxes of 64 head-dim elements by min(page_size, 64) rows.
  CUtensorMap kv_map;
  // The same cache as [K/V][d-half][rows][64] (strides: kv_heads *
  // page_size rows, 128 bytes, one row), one box = a whole 64-key block:
  // K low, K high, V low, V high halves of 64 rows each, the stage layout of
  // the tcgen05 attention.  Set when page_size is a multiple of 64 and
  // head_dim = 128 (AttnArgs::kv4); zero otherwise.
  CUtensorMap kv_map4;
};

// A pointer operand: a fixed plan-owned address, or (slot >= 0) a binding
// slot plus a byte offset.
struct DPtr {
  void* p;
  int slot;
  int pad;
  long long offset;
};

// Device-side error word.  code != 0 after a step means a bounded wait gave
// up or a bounds check failed; info holds (op, cta, where, value).
struct DevStatus {
  unsigned code;
  unsigned info[7];
  unsigned abort;     // set with code: every worker leaves its loop early
  unsigned pad[7];
};

enum DevErr : unsigned {
  DERR_NONE = 0,
  DERR_TIMEOUT = 1,
  DERR_BOUNDS = 2,
  DERR_BAD_OP = 3,
};

// ------------------------------------------------------------------ ops
enum OpKind : int {
  OP_NOP = 0,
  OP_NORM = 1,        // residual add + RMSNorm (+ FP8 quant)
  OP_GEMM = 2,        // weight-streaming projection + fused epilogue
  OP_ATTN = 3,        // split-KV attention + log-sum-exp combine (+ quant)
};

enum Epilogue : int {
  EPI_QKV_ROPE = 0,   // QK-norm + RoPE; q -> buffer, k/v -> paged cache
  EPI_STORE_BF16 = 1, // out[m][n] = bf16(acc)
  EPI_SILU_MUL = 2,   // a = silu(bf16 g) * bf16 u (+ FP8 quant per 128)
  EPI_LOGITS = 3,     // fp32 logits + greedy argmax (lowest index on ties)
  EPI_PARTIALS = 4,   // no fix-up: every CTA publishes its partial of each
                      // tile it touches; the next op (a norm) sums them
};

// Most CTAs whose Stream-K ranges may share one tile of a projection whose
// fix-up the following norm performs (EPI_PARTIALS).
constexpr int kMaxPartContrib = 32;

// L2 prefetch of the first weight tiles the next projection's share with a
// given CTA index will stream (tmap == NULL: none).  Issued by the current
// kernel once its own loads are out, so that the next kernel's first loads
// hit L2.
struct PrefetchSpec {
  const CUtensorMap* tmap;    // the next projection's weights
  int NT, KB, G, t_base, pair, up_row, kel, units;
};

struct NormArgs {
  DPtr x, res;        // bf16 [M, H]
  DPtr r_out;         // bf16 [M, H] new residual
  const void* w;      // bf16 [H]
  void* h_out;        // bf16 [Mp, H] or e4m3 codes [Mp, H]
  float* h_scale;     // FP8: [M, H/128]
  int fp8, M, H, rows_per_cta;
  float eps;
  // The producing projection's Stream-K partials (EPI_PARTIALS), or NULL:
  // x[m][n] = bf16(sum over the CTAs whose ranges hold tile n / 128, in CTA
  // order, of their partial), written to x as well.  Partial slot s holds
  // [part_mp][128] fp32 at part + s * part_mp * 128.
  const float* part;
  int part_U, part_G, part_KB, part_mp;
  // CTAs (shares) per row: a cluster of `split` CTAs each norms a part of
  // the row; in the megakernel share c % split == 0 norms the whole row
  // c / split and the others only pass the dependency
  int split;
};

struct GemmArgs {
  const CUtensorMap* tmap_w;  // weights [N, K], 128B-swizzled boxes (128 B x 128 rows)
  const CUtensorMap* tmap_x;  // activations [Mp, K], boxes (128 B x Mp rows)
  const float* w_scale;       // FP8 block scales [N/128, K/128]
  const float* x_scale;       // FP8 activation scales [M, K/128]
  int fp8;
  int mma;                    // 1: tcgen05 (M > 4), 0: CUDA-core GEMV
  int M, Mp;                  // tokens, rows of the activation tile
  int K;                      // elements
  int KB;                     // 128-byte k-blocks per tile
  int share_max;              // units of the largest CTA share (ceil(NT KB / G))
  int NT;                     // output tiles (pairs for gate/up)
  int t_base;                 // first tile (a branch may cover a sub-range)
  int pair;                   // 1: tile t = gate rows t*128.. + up rows up_row+t*128..
  int up_row;                 // first up row (= I) for gate/up
  int G;                      // CTAs sharing the units
  int stages;
  int tmem_bufs;              // tcgen05 accumulator ring depth
  int epi;
  // partial sums (Stream-K fix-up) and counters
  float* ws;                  // [G][2][npair][Mp][128] fp32
  unsigned* tile_cnt;         // [NT]
  unsigned* done_cnt;         // [1] (EPI_LOGITS)
  // epilogue operands
  DPtr out;                   // STORE_BF16: bf16 [M, ldo]; LOGITS: fp32 [M, V]
  int ldo;
  void* act;                  // SILU_MUL: bf16 [Mp, I] or codes [Mp, I]
  float* act_scale;           // [M, I/128]
  int act_ld;
  // QKV epilogue
  void* q_out;                // bf16 [M, Hq, d]
  DPtr kv, bt, pos;
  const void* q_norm_w;
  const void* k_norm_w;
  const float* rope_cs;       // [max_pos][d/2][2] (cos, sin) fp32
  int rope_max_pos;
  int Hq, Hkv, d, T, P, num_pages, max_pages, layer;
  float eps;
  // LOGITS epilogue
  float* best_val;            // [NT][M]
  int* best_idx;              // [NT][M]
  DPtr ids;                   // int32 [M]
  PrefetchSpec pf;
  // Where a standalone projection waits on its producer (the per-edge
  // programmatic-launch ablation): 0 after issuing its first weight stages
  // (the default), 1 after its prologue but before any load, 2 at kernel
  // entry, before its prologue.
  int gdc_mode;
};

struct AttnArgs {
  DPtr kv, bt, pos;
  const void* q;              // bf16 [M, Hq, d] (after QK-norm + RoPE)
  void* out;                  // bf16 [Mp, Hq d] or codes
  float* out_scale;           // FP8: [M, Hq d / 128]
  int fp8;
  int R, T, Hq, Hkv, d, P, num_pages, max_pages, layer;
  int QR, QRp;                // query rows per pair (T * G), padded to 16
  int NB;                     // 64-key blocks per pair (from max_context)
  int G;                      // CTAs
  int stages;
  int max_ctx;                // positions must lie in [0, max_ctx) (else DERR_BOUNDS)
  int pre_stages;             // > 0: K/V blocks loaded before the dependency wait, at most
  int kv4;                    // 1: a block is one TMA box of Binding::kv_map4
  int split_sm;               // tcgen05 engine: split softmax up to 32 query rows
  float scale_log2;           // log2(e) / sqrt(d)
  float* ws;                  // partials [G][2][QRp][d] + lse [G][2][QRp]
  unsigned* pair_cnt;         // [R * Hkv]
  PrefetchSpec pf;
};

struct OpArgs {
  int kind;
  int pad[3];
  union {
    NormArgs norm;
    GemmArgs gemm;
    AttnArgs attn;
  };
};

// ------------------------------------------------- megakernel instructions
// 32 x u32 = 128 bytes.  Addresses live in the op-argument table, never in
// the instruction; an instruction names its op row and its CTA share.
struct Instr {
  uint32_t op_row;            // index into the OpArgs table (0xffffffff: NoOp)
  uint32_t cta;               // this worker's share index within the op
  uint32_t n_wait;
  uint32_t n_signal;
  uint32_t wait_event[4];
  uint32_t wait_value[4];     // wait until event >= value
  uint32_t signal_event[2];
  uint32_t signal_inc[2];
  uint32_t signal_event_hi[2];  // signals 2 and 3 (n_signal <= 4)
  uint32_t signal_inc_hi[2];
  uint32_t pad[12];
};
static_assert(sizeof(Instr) == 128, "instruction is 128 bytes");

constexpr uint32_t kMaxWaits = 4, kMaxSignals = 4;

__host__ __device__ inline uint32_t instr_signal_event(const Instr& in, uint32_t s) {
  return s < 2 ? in.signal_event[s] : in.signal_event_hi[s - 2];
}
__host__ __device__ inline uint32_t instr_signal_inc(const Instr& in, uint32_t s) {
  return s < 2 ? in.signal_inc[s] : in.signal_inc_hi[s - 2];
}

struct MegaArgs {
  const OpArgs* ops;
  const Instr* queues;        // [workers][qlen]
  int qlen;
  int workers;
  unsigned* events;           // event counters; the last worker to leave
                              // zeroes them (and finish_cnt) for the next step
  unsigned* finish_cnt;
  int num_events;
  unsigned long long budget_ns;
  unsigned* trace;            // optional [workers][qlen][4] (start, ready, done)
  // the worker's shared memory: a ring of `ns` slots of `slot_bytes` at
  // offset 0 (operands, filled by the producer warp in queue order), then
  // the consumers' private area at `priv_off`
  int ns;
  int slot_bytes;
  int priv_off;
};

// Trace build: per (operation, CTA share) kTraceSlots u64 entries.
enum TraceSlot : int {
  TR_START = 0,       // the share's engine starts (after its barrier set-up)
  TR_DEPS = 1,        // its inputs are ready (griddepcontrol / event counters)
  TR_FIRST = 2,       // the first unit's data has reached the consumers
  TR_LOOP_END = 3,    // the last unit of the last run has been consumed
  TR_END = 4,         // the share is done (fix-up / combine / epilogue included)
  TR_UNITS = 5,       // value: work units of the share
  TR_REDUCE = 6,      // the last Stream-K fix-up / split-KV combine it ran ended
  TR_PDEPS = 7,       // megakernel: its producer warp saw the inputs ready
  kTraceSlots = 8
};

struct KernelCtx {
  const Binding* binding;
  DevStatus* status;
  unsigned long long budget_ns;   // bounded-wait budget
  int op_id;                      // for error reports (and the trace row)
  int trace_ctas = 0;             // shares per trace row
  unsigned long long* trace = nullptr;  // [ops][trace_ctas][kTraceSlots] or NULL
};

}  // namespace dl
