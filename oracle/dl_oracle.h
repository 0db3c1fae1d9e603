/*
 * dl_oracle.h -- plain, slow, obviously-correct CPU oracle for one small-batch
 * transformer decode step (Qwen3-shaped layer: add+RMSNorm, QKV projection,
 * QK-norm + RoPE, paged KV write, split-KV GQA attention with log-sum-exp
 * combine, O projection, add+RMSNorm, gate/up + SiLU*mul, down; full steps add
 * the final norm, lm_head and greedy argmax).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this library.  It shares no code, header, table or constant generator with
 * the CUDA library: it is written from the definitions of the operations and
 * is checked against closed forms, invariants, library routines and brute
 * force in tests/test_oracle_*.py.
 *
 * Storage types: bf16 values travel as uint16_t bit patterns, FP8 e4m3 values
 * as uint8_t codes.  All arithmetic is double precision; results are rounded
 * to bf16 (round-to-nearest-even) exactly where the decode step materialises a
 * bf16 tensor.  Where a floating-point value decides an integer (an FP8 code)
 * the decision is taken in fp32, the precision the kernels use.
 *
 * Parity status of each function is stated beside it: "pinned" names the
 * independent check; the two composition functions are pinned through their
 * parts plus structural special cases (zero weights, identity projections);
 * beyond that the whole-layer numbers are "parity unpinned" because no page
 * prints a worked example of a full layer.
 */
#ifndef DL_ORACLE_H
#define DL_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- scalars */

/* bf16 bits -> double (exact).  pinned: torch bfloat16 -> float64 cast. */
double or_bf16_to_double(uint16_t b);
/* double -> bf16 bits, round-to-nearest-even from the exact double value,
 * overflow to +-inf, NaN kept.  pinned: torch float32 -> bfloat16 cast. */
uint16_t or_bf16_from_double(double v);

/* OCP FP8 E4M3FN ("e4m3"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 = NaN, largest finite 448.  pinned: all 256 codes vs
 * torch.float8_e4m3fn. */
double or_e4m3_decode(uint8_t code);
/* Saturating round-to-nearest-even encode: |v| >= 448 -> +-448, NaN -> 0x7F.
 * pinned: every in-range bf16 value vs torch.float8_e4m3fn casts. */
uint8_t or_e4m3_encode(double v);

/* silu(z) = z / (1 + exp(-z)).  pinned: torch.nn.functional.silu float64. */
double or_silu(double z);

/* ------------------------------------------------------------------ ops */

/* Fused residual add + RMSNorm over rows of width H (the decode step's
 * "Add + RMSNorm (+Quant)" step, page "Kernel-Mega-PDL" section 1 and the
 * add_rmsnorm kernel of the gap model on page "PDL and megakernel").
 *   r_out = bf16(x + res);  h = r_out / sqrt(mean(r_out^2) + eps) * w
 * h_bf16 (optional) receives bf16(h); h_f32 (optional) receives (float)h, the
 * value the FP8 path quantises.  pinned: unit-RMS invariant, constant rows. */
void or_add_rmsnorm(int M, int H, const uint16_t* x, const uint16_t* res,
                    const uint16_t* w, double eps, uint16_t* r_out,
                    uint16_t* h_bf16, float* h_f32);

/* Per-token, per-128-group FP8 quantisation (fp32 decisions):
 *   s = amax_g / 448 (s = 1 when amax_g == 0), code = e4m3(v / s).
 * K must be a multiple of 128.  scales is [M, K/128].  pinned: saturation,
 * round trip |code*s - v| <= half an e4m3 step, amax element maps to 448. */
void or_quant_group128(int M, int K, const float* v, uint8_t* codes,
                       float* scales);

/* out[m][n] = sum_k a[m][k] * W[n][k] with W bf16 [N, K] row-major, double
 * accumulation.  pinned: one-hot weights, numpy float64 matmul. */
void or_gemm_bf16(int M, int N, int K, const double* a, const uint16_t* w,
                  double* out);
/* FP8 block-scaled GEMM: a = codes [M, K] with scales [M, K/128]; W = codes
 * [N, K] with scales [N/128, K/128] (one per 128x128 block):
 *   out[m][n] = sum_kb sw[n/128][kb] * sa[m][kb] * sum_{k in kb} dec(w) dec(a)
 * pinned: numpy float64 matmul of the decoded, scaled operands. */
void or_gemm_fp8(int M, int N, int K, const uint8_t* a_codes,
                 const float* a_scales, const uint8_t* w_codes,
                 const float* w_scales, double* out);

/* RMSNorm over one head vector of length d (no residual), times w, in double.
 * pinned: unit-RMS invariant. */
void or_head_rmsnorm(int d, const double* in, const uint16_t* w, double eps,
                     double* out);
/* Rotary embedding, neox half-split pairing (i, i + d/2), at position pos:
 *   inv_freq_i = theta^(-2i/d), angle = pos * inv_freq_i
 *   (x_i, x_j) -> (x_i cos - x_j sin, x_j cos + x_i sin), j = i + d/2.
 * pinned: pair norms preserved, pos 0 is identity, <R_p q, R_s k> depends only
 * on p - s. */
void or_rope(int d, const double* in, int pos, double theta, double* out);

/* Paged KV cache layout [layer][page][2 (K,V)][kv_head][page_size][head_dim].
 * Element offset of (layer, page, kv, head, slot-in-page, dim).
 * pinned: tag round trips, distinct tokens -> distinct slots. */
size_t or_kv_offset(int num_pages, int n_kv_heads, int page_size, int head_dim,
                    int layer, int page, int kv, int head, int slot, int dim);
/* Physical page of logical key position p for request r (block table row r
 * has max_pages entries); returns -1 when out of range. */
int or_kv_page(const int32_t* block_table, int max_pages, int num_pages,
               int page_size, int r, int p);
/* Gather keys or values [0, n_keys) of (request r, kv head h) into dense
 * [n_keys, head_dim] bf16.  kv = 0 keys, 1 values.  Returns 0 or -1. */
int or_kv_gather(const uint16_t* kv_pages, const int32_t* block_table,
                 int max_pages, int num_pages, int n_kv_heads, int page_size,
                 int head_dim, int layer, int r, int h, int kv, int n_keys,
                 uint16_t* out);

/* Softmax attention of one query over keys [k0, k1) of dense K/V rows
 * ([n, d] bf16), scale 1/sqrt(d); keys beyond `last` (causal limit,
 * inclusive) are masked.  Writes the normalised partial output o[d] and its
 * log-sum-exp; an empty range (no unmasked key) gives lse = -inf, o = 0.
 * (Split-KV partial, page "kernel prologue/epilogue" section 4.2.)
 * pinned: one key -> V, equal keys -> mean(V), torch float64 softmax. */
void or_attention_partial(int d, const double* q, const uint16_t* K,
                          const uint16_t* V, int k0, int k1, int last,
                          double* o, double* lse);
/* Log-sum-exp combine of n partials (page "kernel prologue/epilogue" section
 * 4.2): lse = log sum_i exp(lse_i); o = sum_i exp(lse_i - lse) o_i.
 * pinned: equals the unsplit result for any split list (1e-12). */
void or_lse_combine(int d, int n, const double* o_parts,
                    const double* lse_parts, double* o, double* lse);

/* Greedy argmax over n logits; ties resolve to the lowest index.
 * pinned: planted maxima and ties. */
int32_t or_argmax(int n, const float* logits);

/* --------------------------------------------------------- composition */

typedef struct {
  int hidden, inter, n_q_heads, n_kv_heads, head_dim, n_layers, vocab;
  double eps, rope_theta;
  int fp8;                 /* 1: FP8 e4m3 weights + per-token group quant */
  int num_requests, tokens_per_request;
  int page_size, num_pages, max_pages_per_request;
} or_config;

typedef struct {
  const uint16_t* ln1_w;         /* [H] */
  const void* w_qkv;             /* [(Hq+2Hkv)d, H] bf16 or e4m3 codes */
  const float* w_qkv_scale;      /* [N/128, K/128] (FP8 only) */
  const uint16_t* q_norm_w;      /* [d] */
  const uint16_t* k_norm_w;      /* [d] */
  const void* w_o;               /* [H, Hq d] */
  const float* w_o_scale;
  const uint16_t* ln2_w;         /* [H] */
  const void* w_gate_up;         /* [2I, H], rows = [gate | up] */
  const float* w_gate_up_scale;
  const void* w_down;            /* [H, I] */
  const float* w_down_scale;
} or_layer_weights;

/* Optional intermediates of one layer (any pointer may be NULL). */
typedef struct {
  uint16_t* r1;                      /* [M,H] residual after the first add */
  uint16_t* h1;                      /* [M,H] bf16 path */
  uint8_t* h1_codes; float* h1_scales;   /* FP8 path */
  uint16_t* q_rot;                   /* [M, Hq d] after QK-norm + RoPE */
  uint16_t* k_rot;                   /* [M, Hkv d] */
  uint16_t* v;                       /* [M, Hkv d] */
  uint16_t* attn;                    /* [M, Hq d] bf16 path */
  uint8_t* attn_codes; float* attn_scales;
  uint16_t* o2;                      /* [M,H] O projection output */
  uint16_t* r2;                      /* [M,H] residual after the second add */
  uint16_t* h2;
  uint8_t* h2_codes; float* h2_scales;
  uint16_t* act;                     /* [M, I] silu(g)*u */
  uint8_t* act_codes; float* act_scales;
  uint16_t* y;                       /* [M,H] layer output */
} or_layer_trace;

/* One decode layer, definition order (all new K/V of the step are written to
 * the cache before any attention reads it).  Token m belongs to request
 * m / tokens_per_request; positions must be consecutive within a request.
 * Returns 0, or -1 on an invalid argument (page out of range, bad shape). */
int or_decode_layer(const or_config* c, int layer, const or_layer_weights* w,
                    const uint16_t* x, const uint16_t* res, uint16_t* kv_pages,
                    const int32_t* block_table, const int32_t* positions,
                    uint16_t* y_out, uint16_t* r_out, or_layer_trace* trace);

/* Whole step: n_layers layers, then (vocab > 0) final add + RMSNorm, lm_head
 * (bf16 [vocab, H]) into fp32 logits [M, vocab] and greedy ids [M].  With
 * vocab == 0 the step stops after the layers and writes out = [2, M, H]
 * = (y, residual).  trace_last (optional) receives the last layer's
 * intermediates.  Returns 0 or -1. */
int or_decode_step(const or_config* c, const or_layer_weights* layers,
                   const uint16_t* final_norm_w, const uint16_t* lm_head_w,
                   const uint16_t* x, const uint16_t* res, uint16_t* kv_pages,
                   const int32_t* block_table, const int32_t* positions,
                   uint16_t* out, float* logits, int32_t* ids,
                   or_layer_trace* trace_last);

/* Threads the oracle's parallel loops use (OpenMP), for reporting. */
int or_num_threads(void);
void or_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
