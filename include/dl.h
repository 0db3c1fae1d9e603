/*
 * dl.h -- C ABI of the GB300 (sm_103a) small-batch decode-step library.
 *
 * One memory-bound, Qwen3-shaped transformer decode step: fused residual
 * add + RMSNorm (optionally with per-token FP8 quantisation), QKV projection,
 * QK-norm + RoPE, paged KV-cache write, split-KV GQA attention with a
 * log-sum-exp combine, O projection, a second add + RMSNorm, gate/up with
 * SiLU*mul, down projection and, for full steps, the final norm, lm_head and
 * greedy argmax.  The operation list follows the Qwen3 decode kernel list of
 * the gap model on page "PDL and megakernel" (section on estimating the
 * gaps); the fused Add + RMSNorm + Quant step is the first op of page
 * "Kernel-Mega-PDL" (TLDR and section 1); the split-KV combine is page
 * "kernel prologue/epilogue" section 4.2.
 *
 * The step runs under three schedules (page "Kernel-Mega-PDL"):
 *   - serial single-stream kernels (section 1),
 *   - CUDA Graph + multistream branches + programmatic dependent launch, each
 *     consumer prefetching its weights before it waits on its producer
 *     (sections 6 and 7),
 *   - a persistent tile-instruction megakernel, one worker CTA per SM with
 *     host-built per-SM queues and global event counters published with
 *     release adds and awaited with acquire polls (section 4; page "PDL and
 *     megakernel", megakernel section).
 *
 * Conventions.  All pointers passed to dl_decode_step are device pointers
 * (16-byte aligned) unless the name says _host.  bf16 tensors are 16-bit
 * bfloat16 bit patterns; FP8 weights are OCP e4m3 ("E4M3FN") codes with one
 * fp32 scale per 128x128 block.  Weight matrices are [out, in] row-major.
 * Errors: functions return a dl_status; dl_plan_create returns NULL; the
 * message of the last failure on the calling thread is dl_last_error().
 * A plan runs one step at a time: calls on one plan must be ordered by the
 * caller (same stream, or synchronised).
 */
#ifndef DL_H
#define DL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DL_OK = 0,
  DL_ERR_INVALID_ARG = 1,   /* a host-visible argument check failed */
  DL_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
  DL_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  DL_ERR_OOM = 4,           /* device allocation failed */
  DL_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up */
  DL_ERR_PLAN_INVALID = 6,  /* megakernel plan failed host validation */
  DL_ERR_DEVICE_BOUNDS = 7  /* a device-side bounds check failed (bad block
                               table entry or position) */
} dl_status;

typedef enum {
  DL_MODE_SERIAL = 0,            /* one kernel per op, one stream, no PDL */
  DL_MODE_PDL_GRAPH = 1,         /* graph, DAG branches, programmatic edges */
  DL_MODE_MEGAKERNEL = 2,        /* persistent tile-instruction megakernel */
  DL_MODE_GRAPH_LINEAR = 3,      /* graph, linear chain, full edges */
  DL_MODE_GRAPH_LINEAR_PDL = 4,  /* graph, linear chain, programmatic edges */
  DL_MODE_GRAPH_DAG = 5          /* graph, DAG branches, full edges */
} dl_mode;

typedef enum {
  DL_WEIGHT_BF16 = 0,
  DL_WEIGHT_FP8_E4M3_B128 = 1  /* e4m3 codes + fp32 scale per 128x128 block;
                                  activations quantised per token per 128 */
} dl_weight_dtype;

/* Device pointers of one layer's weights.  Caller-owned; they must stay
 * valid and unchanged for the plan's lifetime.  *_scale pointers are [N/128,
 * K/128] fp32 for FP8 weights and NULL for bf16. */
typedef struct {
  const void* ln1_w;        /* bf16 [hidden] */
  const void* w_qkv;        /* [(n_q_heads + 2 n_kv_heads) head_dim, hidden],
                               rows = q heads | k heads | v heads */
  const float* w_qkv_scale;
  const void* q_norm_w;     /* bf16 [head_dim] */
  const void* k_norm_w;     /* bf16 [head_dim] */
  const void* w_o;          /* [hidden, n_q_heads head_dim] */
  const float* w_o_scale;
  const void* ln2_w;        /* bf16 [hidden] */
  const void* w_gate_up;    /* [2 inter, hidden], rows = gate | up */
  const float* w_gate_up_scale;
  const void* w_down;       /* [hidden, inter] */
  const float* w_down_scale;
} dl_layer_weights;

typedef struct {
  int hidden, inter, n_q_heads, n_kv_heads, head_dim, n_layers;
  int vocab;                /* 0: layer plan (no lm_head); else full step */
  float eps;                /* RMSNorm epsilon (inside the square root) */
  float rope_theta;         /* RoPE base; neox half-split pairing */
  int weight_dtype;         /* dl_weight_dtype */
  int num_requests;         /* R */
  int tokens_per_request;   /* T; M = R * T tokens, request-major */
  int page_size;            /* tokens per KV page */
  int num_pages;            /* pages per layer in the cache */
  int max_pages_per_request;/* block-table row length */
  int max_context;          /* largest context (keys) a request may reach */
  int num_sms;              /* worker CTAs; 0 = every SM of the device */
  unsigned modes_mask;      /* bit m: prepare mode m (graphs, queues) */
  const dl_layer_weights* layers;  /* [n_layers], read during create */
  const void* final_norm_w; /* bf16 [hidden] (full steps) */
  const void* lm_head_w;    /* bf16 [vocab, hidden] (full steps) */
} dl_config;

typedef struct dl_plan dl_plan;

/* Build a plan on the current CUDA device: validates cfg, allocates the
 * plan's workspace (activations, split-K/split-KV partials, counters,
 * cos/sin table, TMA descriptors), records the per-mode launch lists,
 * captures the graphs and packs the megakernel queues of modes_mask.
 * Returns NULL on failure (see dl_last_error). */
dl_plan* dl_plan_create(const dl_config* cfg);

/* Message describing the last failure on this thread ("" if none). */
const char* dl_last_error(void);

/* One decode step, asynchronous on `stream` (a cudaStream_t; NULL = legacy
 * default stream).
 *   x, residual  bf16 [M, hidden], read only.
 *   kv_pages     bf16 [n_layers][num_pages][2 (K,V)][n_kv_heads][page_size]
 *                [head_dim]; the step writes K/V of its M tokens in place.
 *   block_table  int32 [num_requests, max_pages_per_request]: logical page
 *                i of request r lives in physical page block_table[r][i].
 *   positions    int32 [M]: token m of request r = m / T sits at this
 *                position; positions of a request are consecutive and its
 *                context after the step is positions[last] + 1 keys.
 *   out          layer plans: bf16 [2, M, hidden] = (layer output, new
 *                residual); full plans: int32 [M] greedy token ids.
 * Host-checkable errors return synchronously (DL_ERR_INVALID_ARG).
 * Device-side failures (bounded wait expiry, bad block-table entry) are
 * reported by dl_plan_status after the stream is synchronised. */
dl_status dl_decode_step(dl_plan* plan, const void* x, const void* residual,
                         void* kv_pages, const int32_t* block_table,
                         const int32_t* positions, void* out, int mode,
                         void* stream);

/* End-to-end variant: x, residual, block_table, positions and out are HOST
 * buffers; kv_pages is a device pointer.  When all five host buffers are
 * device-addressable page-locked memory (cudaHostAlloc / cudaHostRegister,
 * mapped under unified addressing, 16-byte aligned) the kernels read the
 * inputs and write the result across the host link in place, with no copy
 * of their own; otherwise the step copies them to and from plan-owned
 * device buffers on `stream` (asynchronous for page-locked buffers).  The
 * result is in out_host once the stream is done. */
dl_status dl_decode_step_host(dl_plan* plan, const void* x_host,
                              const void* residual_host, void* kv_pages,
                              const int32_t* block_table_host,
                              const int32_t* positions_host, void* out_host,
                              int mode, void* stream);

/* Device-side status of the last step(s); call after synchronising.  Reading
 * it clears it. */
dl_status dl_plan_status(dl_plan* plan);

/* Trace build.  A plan created while the environment holds DL_TRACE=1
 * records, for every CTA share of every operation it runs, %globaltimer
 * stamps in nanoseconds (the in-kernel timeline the megakernel section of
 * page "Kernel-Mega-PDL" reads its active-SM curve from):
 *   [0] share starts  [1] inputs ready  [2] first unit's data consumed
 *   [3] last unit consumed  [4] share done  [5] work units (a count, not a
 *   time)  [6] end of the last Stream-K fix-up / split-KV combine the share
 *   ran (0 if none)  [7] unused.
 * Table layout: uint64 [n_ops][n_ctas][8]; op i is op i of the serial list
 * (dl_plan_op_info) in the serial, linear-graph and megakernel schedules,
 * and node i of the branch list in the DAG schedules.  dl_plan_trace
 * reports the dimensions (either pointer may be NULL); with host_buf it
 * synchronises the device, copies the table (bytes >= n_ops * n_ctas * 64)
 * and clears it.  DL_ERR_UNSUPPORTED for a plan created without tracing.
 * Tracing costs one predicated branch per stamp when off. */
dl_status dl_plan_trace(dl_plan* plan, void* host_buf, size_t bytes,
                        int* n_ops, int* n_ctas);

/* fp32 logits [M, vocab] of the last full step (device pointer), or NULL. */
const float* dl_plan_logits(dl_plan* plan);

/* Debug access to a plan-owned intermediate buffer of the last layer run:
 *   0 r1 (bf16 [M,H])     1 h1 (bf16 [Mp,H] or e4m3 [Mp,H])  2 h1 scales
 *   3 q (bf16 [M,Hq,d])   4 attn (bf16/e4m3 [Mp, Hq d])       5 attn scales
 *   6 o2 (bf16 [M,H])     7 r2 (bf16 [M,H])                   8 h2
 *   9 h2 scales           10 act (bf16/e4m3 [Mp, I])          11 act scales
 *   12 y (bf16 [M,H])     16 final RMSNorm output, the lm_head input (bf16
 *                          [M,H]; full-step plans only)
 * Returns DL_ERR_INVALID_ARG for an unknown index. */
dl_status dl_plan_debug_buffer(dl_plan* plan, int which, void** ptr,
                               size_t* bytes);

/* Number of kernels one step of `mode` launches (for accounting). */
int dl_plan_kernel_count(dl_plan* plan, int mode);

/* The serial schedule's operations: how many, the name of op i, and a
 * launch of op i alone on `stream` (for per-kernel timing; operands are
 * those bound by the last dl_decode_step on this plan).  dl_plan_op_info
 * also reports the op's grid (CTAs) and dynamic shared memory bytes. */
int dl_plan_op_count(dl_plan* plan);
dl_status dl_plan_op_info(dl_plan* plan, int i, char* name, size_t name_len,
                          int* grid, int* smem_bytes);
dl_status dl_plan_launch_op(dl_plan* plan, int i, void* stream);

/* The serial schedule's operations [first, first + count) launched in order
 * on `stream`, with programmatic stream serialization on every launch when
 * `pdl` != 0, and every projection waiting on its producer where `gdc_mode`
 * says: 0 after issuing its first weight stages (the schedules' own
 * placement), 1 after its prologue (barriers, TMEM, descriptors) but before
 * any load, 2 at kernel entry.  A measurement hook for the per-edge ablation
 * of programmatic dependent launch (page "Kernel-Mega-PDL", the section on
 * where the gain of PDL comes from: its entry / deepgemm / prefetch
 * consumers); captured in a
 * CUDA graph it gives the producer-start to consumer-end span of an edge.
 * Operands are those bound by the last dl_decode_step on this plan.
 * DL_ERR_INVALID_ARG for a bad range or mode, or before any step. */
dl_status dl_plan_launch_ops(dl_plan* plan, int first, int count, int pdl, int gdc_mode,
                             void* stream);

/* Megakernel queue statistics: workers, queue length, events. */
dl_status dl_plan_mega_info(dl_plan* plan, int* workers, int* qlen,
                            int* events);

/* Test hook for failure detection: with `delta` != 0 the megakernel plan's
 * first wait threshold is raised by delta WITHOUT host validation, so the
 * device wait must expire (bounded by budget_ns) and report DL_ERR_TIMEOUT.
 * delta = 0 restores the validated plan.  Returns DL_ERR_PLAN_INVALID if the
 * validator rejects the modified plan when validate != 0. */
dl_status dl_plan_debug_perturb_wait(dl_plan* plan, unsigned delta,
                                     unsigned long long budget_ns,
                                     int validate);

void dl_plan_destroy(dl_plan* plan);

/* ------------------------------------------- attention without allocation
 * The split-KV GQA attention of one layer (per (request, kv head) the keys
 * are split over CTAs, each partial keeps its rows' log-sum-exp, and once
 * every partial of a pair is published each CTA of the pair combines a
 * slice of its query rows), for callers that may not allocate device memory
 * where they call it: a framework that owns the device allocator and forbids
 * foreign allocations, or code running under a memory-pool budget that is
 * already spent.  The paper has no counterpart of this entry point.  It
 * launches the split-KV attention kernel of the mma.sync engine (the
 * megakernel's attention engine) with the plans' work split and pipeline
 * depth.  It allocates nothing, neither through CUDA nor through a library:
 * its binding table, status word, arrival counters and fp32 partials live in
 * one statically reserved 8 MiB device array, which every GPU that loads the
 * library holds until exit.
 *
 *   cfg          only the attention fields are read: n_q_heads, n_kv_heads,
 *                head_dim (128), n_layers, weight_dtype (FP8 selects e4m3
 *                output), num_requests, tokens_per_request, page_size,
 *                num_pages, max_pages_per_request, max_context, num_sms.
 *   layer        which layer of the cache to attend over.
 *   q            bf16 [M, n_q_heads, head_dim], after QK-norm and RoPE.
 *   kv_pages, block_table, positions  as in dl_decode_step; the cache must
 *                already hold this step's K/V (it is only read here).
 *                Every position must lie in [0, max_context).
 *   out          bf16 [M, n_q_heads head_dim]; with FP8, e4m3 codes of the
 *                same shape plus out_scale fp32 [M, n_q_heads head_dim / 128]
 *                (one scale per token per 128 values; NULL for bf16).
 *   check        0: asynchronous on `stream`; nonzero: also synchronise the
 *                stream and report device-side failures (DL_ERR_TIMEOUT;
 *                DL_ERR_DEVICE_BOUNDS for a position outside [0,
 *                max_context) or a block-table entry outside [0,
 *                num_pages), after which the output is unspecified).
 * Limits: the partials take G x 2 x QRp x 516 bytes of the 8 MiB.  QRp is
 * tokens_per_request x group size rounded up to 16, 32 or 64.  G is the
 * CTA count of the split (the plans' rule without their minimum of four
 * blocks a CTA): with pairs = num_requests x n_kv_heads, blocks =
 * ceil(max_context / 64) and S = num_sms (0: every SM), G = min(pairs x
 * min(62, S / pairs), pairs x blocks) when pairs <= S, else min(S, pairs x
 * blocks); it is at most S.  num_requests x n_kv_heads <= 4096.  Larger
 * requests are rejected with DL_ERR_UNSUPPORTED and a message naming the
 * bytes needed (on a 152-SM GPU, QRp = 64 needs num_sms <= 126).  All
 * tensor pointers are caller-owned.
 * Set-up: the first call on a device (made with that device current) looks
 * up the scratch's device address and sets the kernels' shared-memory
 * limit; make that first call before any stream capture.
 * Concurrency: every call on a device uses the same scratch, which keeps the
 * last call's contents; the call clears what must start at zero.  Calls
 * whose GPU work may overlap in time (other streams, other threads) race
 * and corrupt each other's results: order them on one stream or
 * synchronise. */
dl_status dl_attention_noalloc(const dl_config* cfg, int layer, const void* q,
                               const void* kv_pages, const int32_t* block_table,
                               const int32_t* positions, void* out,
                               float* out_scale, int check, void* stream);

/* ------------------------------------------------------- measurement
 * Microbenchmarks of the mechanisms the schedules rest on, each one small
 * synchronous run on the current device (they allocate a few bytes of
 * device memory, and return DL_ERR_TIMEOUT if a bounded device wait gave
 * up).
 *   dl_bench_mma: one CTA issues n_mma tcgen05.mma instructions (M = 128,
 *     N = n in 16..256, a multiple of 16; fp8 != 0: kind::f8f6f4 e4m3 with
 *     K = 32, else kind::f16 bf16 with K = 16) over zero operands in shared
 *     memory, into n_accumulators TMEM accumulators (n_accumulators x n <=
 *     512) in turn, from n_issuers (1 or 2) threads; *ns_per_mma = the span
 *     from the first issue to the completion of the last, over n_mma (a
 *     multiple of 4, <= 65536).  lean = 0: each MMA's descriptors and
 *     accumulator are computed in the loop, as a straightforward issuer
 *     does; lean != 0: descriptors built once and advanced by constants,
 *     four MMAs per pass into one accumulator per issuer.  The cost of the
 *     projections' and attention's tensor-core work at the decode step's
 *     small N.
 *   dl_bench_poll_latency: two co-resident CTAs pass a token back and forth
 *     through one global counter, red.release.gpu.add on one side,
 *     ld.acquire.gpu polling on the other (the megakernel's event protocol,
 *     page "Kernel-Mega-PDL", section 4); *ns_per_round_trip over iters
 *     (<= 2^20) round trips.
 *   dl_plan_bench_empty_megakernel: the plan's megakernel launched iters
 *     times on `stream` with every worker's queue a single NoOp: the cost
 *     of the framework itself (page "Kernel-Mega-PDL", the megakernel's
 *     empty-framework run); *us_per_launch from CUDA events.  Needs a plan
 *     built with the megakernel mode; synchronises the stream. */
dl_status dl_bench_mma(int fp8, int n, int n_mma, int n_accumulators, int n_issuers,
                       int lean, double* ns_per_mma);
dl_status dl_bench_poll_latency(int iters, double* ns_per_round_trip);
dl_status dl_plan_bench_empty_megakernel(dl_plan* plan, int iters, double* us_per_launch,
                                         void* stream);

/* ------------------------------------------------------ test-only exports
 * Bit-exact paged-KV indexing (the slot math of the QKV epilogue and the
 * block-table gather of attention) as pure copies:
 *   dl_test_kv_write: for each token m (request m / T, position positions[m])
 *     copy src[m][kv][h][0..d) to kv_pages[layer][page][kv][h][slot][...]
 *     with page = block_table[r][p / P], slot = p % P.
 *   dl_test_kv_gather: dst[r][kv][h][j][0..d) = the cache row of key j of
 *     request r, j < n_keys (same mapping).
 * All pointers device; the calls are asynchronous on `stream`. */
dl_status dl_test_kv_write(const void* src, void* kv_pages,
                           const int32_t* block_table,
                           const int32_t* positions, int layer, int M, int T,
                           int n_kv_heads, int head_dim, int page_size,
                           int num_pages, int max_pages, void* stream);
dl_status dl_test_kv_gather(const void* kv_pages, const int32_t* block_table,
                            void* dst, int layer, int R, int n_keys,
                            int n_kv_heads, int head_dim, int page_size,
                            int num_pages, int max_pages, void* stream);

/* Megakernel queue validator (page "Kernel-Mega-PDL", section 4: a wait
 * may name only an event of an earlier instruction in the global order, so
 * the persistent grid cannot deadlock), on a host description:
 *   queues: host array [workers][qlen] of 128-byte instructions, each 32
 *     uint32: op_row (0xffffffff = NoOp), cta, n_wait (<= 4), n_signal
 *     (<= 2), wait_event[4], wait_value[4], signal_event[2],
 *     signal_inc[2], 16 unused words.
 * DL_OK when every queue lists its ops in increasing op_row, ends with at
 * least one NoOp and has nothing after it, and every wait names an event
 * e < its own op_row whose total signal increments over all queues reach
 * the awaited value; otherwise DL_ERR_PLAN_INVALID with a message
 * (dl_last_error).  DL_ERR_INVALID_ARG for a NULL or empty description.
 * Pure host code: no device is touched. */
dl_status dl_test_validate_mega_queues(const void* queues, int workers, int qlen,
                                       int n_events);

#ifdef __cplusplus
}
#endif
#endif /* DL_H */
