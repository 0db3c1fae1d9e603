/*
 * dl_oracle.c -- CPU oracle for the decode step.  TEST INFRASTRUCTURE ONLY:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg use it.
 * See dl_oracle.h for the contract and the parity status of each function.
 *
 * Written from the definitions of the operations:
 *   - residual add + RMSNorm (+ per-token FP8 quant): page "Kernel-Mega-PDL",
 *     sections TLDR and 1 (Add + RMSNorm + Quant); page "PDL and megakernel",
 *     gap-model kernel list (add_rmsnorm).
 *   - QKV / O / gate-up / down projections, QK-norm + RoPE, KV cache write,
 *     attention, SiLU*mul, final norm, lm_head, sample: page "PDL and
 *     megakernel", gap-model kernel list (Qwen3 decode step).
 *   - split-KV partials and the log-sum-exp combine: page "kernel
 *     prologue/epilogue", section 4.2 (w_i = exp(lse_i - lse)).
 *   - paged KV with a block table: page "Kernel-Mega-PDL", section 4
 *     (OperandPtrTable row of the paged score op: context_lens, block_table).
 */
#include "dl_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------- scalars */

double or_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round-half-to-even of a non-negative double to an integer-valued double. */
static double rne_nonneg(double q) {
  double f = floor(q);
  double r = q - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

uint16_t or_bf16_from_double(double v) {
  if (isnan(v)) return (uint16_t)0x7FC0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  double r;
  if (a == 0.0) {
    r = 0.0;
  } else if (a < ldexp(1.0, -126)) {
    /* bf16 subnormals: quantum 2^-133 */
    r = rne_nonneg(a / ldexp(1.0, -133)) * ldexp(1.0, -133);
  } else {
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    /* 8 significant bits (1 implicit + 7 stored): m * 2^8 in [128, 256) */
    r = ldexp(rne_nonneg(ldexp(m, 8)), e - 8);
  }
  float f;
  if (r > 3.3895313892515355e38) {
    f = INFINITY;
  } else {
    f = (float)r; /* exact: r has at most 8 significant bits */
  }
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t b = (uint16_t)(u >> 16);
  if (neg) b |= 0x8000;
  return b;
}

double or_e4m3_decode(uint8_t code) {
  int s = code >> 7;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

uint8_t or_e4m3_encode(double v) {
  if (isnan(v)) return 0x7F;
  uint8_t s = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a >= 448.0) return (uint8_t)(s | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: quantum 2^-9; 8 quanta is the smallest normal */
    int n = (int)rne_nonneg(a / ldexp(1.0, -9));
    return (uint8_t)(s | n); /* n == 8 encodes exponent field 1, mantissa 0 */
  }
  int e;
  double m = frexp(a, &e); /* a = m 2^e, m in [0.5,1) -> a = (2m) 2^(e-1) */
  int ex = e - 1;          /* unbiased exponent, -6 .. 8 */
  int n = (int)rne_nonneg((2.0 * m - 1.0) * 8.0);
  if (n == 8) {
    n = 0;
    ex += 1;
  }
  if (ex > 8 || (ex == 8 && n > 6)) return (uint8_t)(s | 0x7E);
  return (uint8_t)(s | ((ex + 7) << 3) | n);
}

double or_silu(double z) { return z / (1.0 + exp(-z)); }

/* ----------------------------------------------------------------- ops */

void or_add_rmsnorm(int M, int H, const uint16_t* x, const uint16_t* res,
                    const uint16_t* w, double eps, uint16_t* r_out,
                    uint16_t* h_bf16, float* h_f32) {
  double* r = (double*)malloc(sizeof(double) * (size_t)H);
  for (int m = 0; m < M; ++m) {
    double ss = 0.0;
    for (int i = 0; i < H; ++i) {
      size_t o = (size_t)m * H + i;
      uint16_t rb = or_bf16_from_double(or_bf16_to_double(x[o]) +
                                        or_bf16_to_double(res[o]));
      if (r_out) r_out[o] = rb;
      r[i] = or_bf16_to_double(rb); /* the norm reads the stored residual */
      ss += r[i] * r[i];
    }
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; ++i) {
      size_t o = (size_t)m * H + i;
      double h = r[i] * inv * or_bf16_to_double(w[i]);
      if (h_bf16) h_bf16[o] = or_bf16_from_double(h);
      if (h_f32) h_f32[o] = (float)h;
    }
  }
  free(r);
}

void or_quant_group128(int M, int K, const float* v, uint8_t* codes,
                       float* scales) {
  int G = K / 128;
  for (int m = 0; m < M; ++m) {
    for (int g = 0; g < G; ++g) {
      const float* src = v + (size_t)m * K + (size_t)g * 128;
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i) {
        float a = fabsf(src[i]);
        if (a > amax) amax = a;
      }
      float s = amax > 0.0f ? amax / 448.0f : 1.0f; /* fp32 division */
      scales[(size_t)m * G + g] = s;
      for (int i = 0; i < 128; ++i) {
        float q = src[i] / s; /* fp32 division: the kernels' precision */
        codes[(size_t)m * K + (size_t)g * 128 + i] = or_e4m3_encode((double)q);
      }
    }
  }
}

void or_gemm_bf16(int M, int N, int K, const double* a, const uint16_t* w,
                  double* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint16_t* wr = w + (size_t)n * K;
    for (int m = 0; m < M; ++m) {
      const double* ar = a + (size_t)m * K;
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += ar[k] * or_bf16_to_double(wr[k]);
      out[(size_t)m * N + n] = acc;
    }
  }
}

void or_gemm_fp8(int M, int N, int K, const uint8_t* a_codes,
                 const float* a_scales, const uint8_t* w_codes,
                 const float* w_scales, double* out) {
  int KB = K / 128;
  double lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = or_e4m3_decode((uint8_t)c);
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint8_t* wr = w_codes + (size_t)n * K;
    for (int m = 0; m < M; ++m) {
      const uint8_t* ar = a_codes + (size_t)m * K;
      double acc = 0.0;
      for (int kb = 0; kb < KB; ++kb) {
        double blk = 0.0;
        for (int k = kb * 128; k < kb * 128 + 128; ++k)
          blk += lut[wr[k]] * lut[ar[k]];
        acc += (double)w_scales[(size_t)(n / 128) * KB + kb] *
               (double)a_scales[(size_t)m * KB + kb] * blk;
      }
      out[(size_t)m * N + n] = acc;
    }
  }
}

void or_head_rmsnorm(int d, const double* in, const uint16_t* w, double eps,
                     double* out) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += in[i] * in[i];
  double inv = 1.0 / sqrt(ss / d + eps);
  for (int i = 0; i < d; ++i) out[i] = in[i] * inv * or_bf16_to_double(w[i]);
}

void or_rope(int d, const double* in, int pos, double theta, double* out) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * i / d);
    double ang = (double)pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    double xi = in[i], xj = in[i + half];
    out[i] = xi * c - xj * s;
    out[i + half] = xj * c + xi * s;
  }
}

size_t or_kv_offset(int num_pages, int n_kv_heads, int page_size, int head_dim,
                    int layer, int page, int kv, int head, int slot, int dim) {
  size_t o = (size_t)layer;
  o = o * (size_t)num_pages + (size_t)page;
  o = o * 2 + (size_t)kv;
  o = o * (size_t)n_kv_heads + (size_t)head;
  o = o * (size_t)page_size + (size_t)slot;
  o = o * (size_t)head_dim + (size_t)dim;
  return o;
}

int or_kv_page(const int32_t* block_table, int max_pages, int num_pages,
               int page_size, int r, int p) {
  if (p < 0) return -1;
  int lp = p / page_size;
  if (lp >= max_pages) return -1;
  int32_t pg = block_table[(size_t)r * max_pages + lp];
  if (pg < 0 || pg >= num_pages) return -1;
  return pg;
}

int or_kv_gather(const uint16_t* kv_pages, const int32_t* block_table,
                 int max_pages, int num_pages, int n_kv_heads, int page_size,
                 int head_dim, int layer, int r, int h, int kv, int n_keys,
                 uint16_t* out) {
  for (int j = 0; j < n_keys; ++j) {
    int pg = or_kv_page(block_table, max_pages, num_pages, page_size, r, j);
    if (pg < 0) return -1;
    size_t base = or_kv_offset(num_pages, n_kv_heads, page_size, head_dim,
                               layer, pg, kv, h, j % page_size, 0);
    memcpy(out + (size_t)j * head_dim, kv_pages + base,
           sizeof(uint16_t) * (size_t)head_dim);
  }
  return 0;
}

void or_attention_partial(int d, const double* q, const uint16_t* K,
                          const uint16_t* V, int k0, int k1, int last,
                          double* o, double* lse) {
  int hi = k1 < last + 1 ? k1 : last + 1;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (hi <= k0) {
    *lse = -INFINITY;
    return;
  }
  int n = hi - k0;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    const uint16_t* kr = K + (size_t)(k0 + j) * d;
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += q[i] * or_bf16_to_double(kr[i]);
    s[j] = acc * scale;
    if (s[j] > mx) mx = s[j];
  }
  double l = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = exp(s[j] - mx);
    l += s[j];
  }
  for (int j = 0; j < n; ++j) {
    const uint16_t* vr = V + (size_t)(k0 + j) * d;
    double p = s[j] / l;
    for (int i = 0; i < d; ++i) o[i] += p * or_bf16_to_double(vr[i]);
  }
  *lse = mx + log(l);
  free(s);
}

void or_lse_combine(int d, int n, const double* o_parts,
                    const double* lse_parts, double* o, double* lse) {
  double mx = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (lse_parts[i] > mx) mx = lse_parts[i];
  for (int k = 0; k < d; ++k) o[k] = 0.0;
  if (mx == -INFINITY) {
    *lse = -INFINITY;
    return;
  }
  double sum = 0.0;
  for (int i = 0; i < n; ++i) sum += exp(lse_parts[i] - mx);
  double L = mx + log(sum);
  for (int i = 0; i < n; ++i) {
    double wgt = exp(lse_parts[i] - L); /* empty split: exp(-inf) = 0 */
    for (int k = 0; k < d; ++k) o[k] += wgt * o_parts[(size_t)i * d + k];
  }
  *lse = L;
}

int32_t or_argmax(int n, const float* logits) {
  int32_t best = 0;
  for (int i = 1; i < n; ++i)
    if (logits[i] > logits[best]) best = i; /* strict: ties keep the lowest */
  return best;
}

/* --------------------------------------------------------- composition */

static void round_bf16_array(size_t n, const double* in, uint16_t* out) {
  for (size_t i = 0; i < n; ++i) out[i] = or_bf16_from_double(in[i]);
}

static void bf16_to_double_array(size_t n, const uint16_t* in, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = or_bf16_to_double(in[i]);
}

/* Projection of the activation (bf16 or FP8 codes+scales) by W. */
static void project(const or_config* c, int M, int N, int K,
                    const uint16_t* a_bf16, const uint8_t* a_codes,
                    const float* a_scales, const void* w, const float* w_scale,
                    double* out) {
  if (c->fp8) {
    or_gemm_fp8(M, N, K, a_codes, a_scales, (const uint8_t*)w, w_scale, out);
  } else {
    double* a = (double*)malloc(sizeof(double) * (size_t)M * K);
    bf16_to_double_array((size_t)M * K, a_bf16, a);
    or_gemm_bf16(M, N, K, a, (const uint16_t*)w, out);
    free(a);
  }
}

int or_decode_layer(const or_config* c, int layer, const or_layer_weights* w,
                    const uint16_t* x, const uint16_t* res, uint16_t* kv_pages,
                    const int32_t* block_table, const int32_t* positions,
                    uint16_t* y_out, uint16_t* r_out, or_layer_trace* t) {
  const int H = c->hidden, I = c->inter, Hq = c->n_q_heads,
            Hkv = c->n_kv_heads, d = c->head_dim;
  const int R = c->num_requests, T = c->tokens_per_request, M = R * T;
  const int G = Hq / Hkv, P = c->page_size;
  const int NQKV = (Hq + 2 * Hkv) * d;
  if (Hkv <= 0 || Hq % Hkv != 0 || d % 2 != 0) return -1;
  if (c->fp8 && (H % 128 || I % 128 || (Hq * d) % 128 || NQKV % 128))
    return -1;
  /* positions must be consecutive inside each request */
  for (int r = 0; r < R; ++r)
    for (int t = 1; t < T; ++t)
      if (positions[r * T + t] != positions[r * T + t - 1] + 1) return -1;

  int rc = -1;
  uint16_t* r1 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
  uint16_t* h1 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
  float* hf = (float*)malloc(sizeof(float) * (size_t)M * H);
  const int KMAX = I > H ? (I > Hq * d ? I : Hq * d) : (H > Hq * d ? H : Hq * d);
  uint8_t* codes = (uint8_t*)malloc((size_t)M * KMAX);
  float* scl = (float*)malloc(sizeof(float) * (size_t)M * (KMAX / 128 + 1));
  double* qkv = (double*)malloc(sizeof(double) * (size_t)M * NQKV);
  uint16_t* qrot = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * Hq * d);
  double* attn = (double*)malloc(sizeof(double) * (size_t)M * Hq * d);
  uint16_t* attn_b = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * Hq * d);
  float* attn_f = (float*)malloc(sizeof(float) * (size_t)M * Hq * d);
  double* proj = (double*)malloc(sizeof(double) * (size_t)M * (2 * I > H ? 2 * I : H));
  uint16_t* o2 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
  uint16_t* r2 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
  uint16_t* h2 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * H);
  uint16_t* act = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * I);
  float* act_f = (float*)malloc(sizeof(float) * (size_t)M * I);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)d * 2);

  /* 1. residual add + RMSNorm (+ per-token FP8 quant) */
  or_add_rmsnorm(M, H, x, res, w->ln1_w, c->eps, r1, h1, hf);
  if (c->fp8) or_quant_group128(M, H, hf, codes, scl);
  if (t && t->r1) memcpy(t->r1, r1, sizeof(uint16_t) * (size_t)M * H);
  if (t && t->h1 && !c->fp8) memcpy(t->h1, h1, sizeof(uint16_t) * (size_t)M * H);
  if (t && c->fp8 && t->h1_codes) memcpy(t->h1_codes, codes, (size_t)M * H);
  if (t && c->fp8 && t->h1_scales)
    memcpy(t->h1_scales, scl, sizeof(float) * (size_t)M * (H / 128));

  /* 2. QKV projection, rounded to bf16 */
  project(c, M, NQKV, H, h1, codes, scl, w->w_qkv, w->w_qkv_scale, qkv);
  for (size_t i = 0; i < (size_t)M * NQKV; ++i)
    qkv[i] = or_bf16_to_double(or_bf16_from_double(qkv[i]));

  /* 3-4. QK-norm + RoPE; write k and v of every new token into the cache */
  for (int m = 0; m < M; ++m) {
    int r = m / T, pos = positions[m];
    for (int hh = 0; hh < Hq + Hkv; ++hh) {
      const double* src = qkv + (size_t)m * NQKV + (size_t)hh * d;
      const uint16_t* nw = hh < Hq ? w->q_norm_w : w->k_norm_w;
      or_head_rmsnorm(d, src, nw, c->eps, tmp);
      for (int i = 0; i < d; ++i) tmp[i] = or_bf16_to_double(or_bf16_from_double(tmp[i]));
      or_rope(d, tmp, pos, c->rope_theta, tmp + d);
      if (hh < Hq) {
        round_bf16_array((size_t)d, tmp + d, qrot + (size_t)m * Hq * d + (size_t)hh * d);
      } else {
        int kh = hh - Hq;
        int pg = or_kv_page(block_table, c->max_pages_per_request, c->num_pages, P, r, pos);
        if (pg < 0) goto done;
        size_t ko = or_kv_offset(c->num_pages, Hkv, P, d, layer, pg, 0, kh, pos % P, 0);
        size_t vo = or_kv_offset(c->num_pages, Hkv, P, d, layer, pg, 1, kh, pos % P, 0);
        const double* vsrc = qkv + (size_t)m * NQKV + (size_t)(Hq + Hkv + kh) * d;
        for (int i = 0; i < d; ++i) {
          uint16_t kb = or_bf16_from_double(tmp[d + i]);
          kv_pages[ko + i] = kb;
          kv_pages[vo + i] = or_bf16_from_double(vsrc[i]);
          if (t && t->k_rot) t->k_rot[(size_t)m * Hkv * d + (size_t)kh * d + i] = kb;
          if (t && t->v) t->v[(size_t)m * Hkv * d + (size_t)kh * d + i] = kv_pages[vo + i];
        }
      }
    }
  }
  if (t && t->q_rot) memcpy(t->q_rot, qrot, sizeof(uint16_t) * (size_t)M * Hq * d);

  /* 5-6. attention over keys [0, pos] of each token (after all writes) */
  {
    int fail = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : fail)
    for (int mh = 0; mh < M * Hq; ++mh) {
      int m = mh / Hq, hq = mh % Hq, r = m / T, pos = positions[m];
      int n = pos + 1;
      uint16_t* K = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
      uint16_t* V = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
      double* q = (double*)malloc(sizeof(double) * (size_t)d);
      double lse;
      if (or_kv_gather(kv_pages, block_table, c->max_pages_per_request, c->num_pages, Hkv, P, d,
                       layer, r, hq / G, 0, n, K) ||
          or_kv_gather(kv_pages, block_table, c->max_pages_per_request, c->num_pages, Hkv, P, d,
                       layer, r, hq / G, 1, n, V)) {
        fail = 1;
      } else {
        for (int i = 0; i < d; ++i)
          q[i] = or_bf16_to_double(qrot[(size_t)m * Hq * d + (size_t)hq * d + i]);
        or_attention_partial(d, q, K, V, 0, n, pos, attn + (size_t)m * Hq * d + (size_t)hq * d,
                             &lse);
      }
      free(K);
      free(V);
      free(q);
    }
    if (fail) goto done;
  }
  for (size_t i = 0; i < (size_t)M * Hq * d; ++i) {
    attn_b[i] = or_bf16_from_double(attn[i]);
    attn_f[i] = (float)attn[i];
  }
  if (c->fp8) or_quant_group128(M, Hq * d, attn_f, codes, scl);
  if (t && t->attn && !c->fp8) memcpy(t->attn, attn_b, sizeof(uint16_t) * (size_t)M * Hq * d);
  if (t && c->fp8 && t->attn_codes) memcpy(t->attn_codes, codes, (size_t)M * Hq * d);
  if (t && c->fp8 && t->attn_scales)
    memcpy(t->attn_scales, scl, sizeof(float) * (size_t)M * (Hq * d / 128));

  /* 7. O projection; 8. residual add + RMSNorm (+ quant) */
  project(c, M, H, Hq * d, attn_b, codes, scl, w->w_o, w->w_o_scale, proj);
  round_bf16_array((size_t)M * H, proj, o2);
  if (t && t->o2) memcpy(t->o2, o2, sizeof(uint16_t) * (size_t)M * H);
  or_add_rmsnorm(M, H, o2, r1, w->ln2_w, c->eps, r2, h2, hf);
  if (c->fp8) or_quant_group128(M, H, hf, codes, scl);
  if (t && t->r2) memcpy(t->r2, r2, sizeof(uint16_t) * (size_t)M * H);
  if (t && t->h2 && !c->fp8) memcpy(t->h2, h2, sizeof(uint16_t) * (size_t)M * H);
  if (t && c->fp8 && t->h2_codes) memcpy(t->h2_codes, codes, (size_t)M * H);
  if (t && c->fp8 && t->h2_scales)
    memcpy(t->h2_scales, scl, sizeof(float) * (size_t)M * (H / 128));

  /* 9. gate/up projection, a = silu(bf16 g) * bf16 u (+ quant) */
  project(c, M, 2 * I, H, h2, codes, scl, w->w_gate_up, w->w_gate_up_scale, proj);
  for (int m = 0; m < M; ++m)
    for (int j = 0; j < I; ++j) {
      double g = or_bf16_to_double(or_bf16_from_double(proj[(size_t)m * 2 * I + j]));
      double u = or_bf16_to_double(or_bf16_from_double(proj[(size_t)m * 2 * I + I + j]));
      double a = or_silu(g) * u;
      act[(size_t)m * I + j] = or_bf16_from_double(a);
      act_f[(size_t)m * I + j] = (float)a;
    }
  if (c->fp8) or_quant_group128(M, I, act_f, codes, scl);
  if (t && t->act && !c->fp8) memcpy(t->act, act, sizeof(uint16_t) * (size_t)M * I);
  if (t && c->fp8 && t->act_codes) memcpy(t->act_codes, codes, (size_t)M * I);
  if (t && c->fp8 && t->act_scales)
    memcpy(t->act_scales, scl, sizeof(float) * (size_t)M * (I / 128));

  /* 10. down projection */
  project(c, M, H, I, act, codes, scl, w->w_down, w->w_down_scale, proj);
  round_bf16_array((size_t)M * H, proj, y_out);
  memcpy(r_out, r2, sizeof(uint16_t) * (size_t)M * H);
  if (t && t->y) memcpy(t->y, y_out, sizeof(uint16_t) * (size_t)M * H);
  rc = 0;

done:
  free(r1); free(h1); free(hf); free(codes); free(scl); free(qkv); free(qrot);
  free(attn); free(attn_b); free(attn_f); free(proj); free(o2); free(r2);
  free(h2); free(act); free(act_f); free(tmp);
  return rc;
}

int or_decode_step(const or_config* c, const or_layer_weights* layers,
                   const uint16_t* final_norm_w, const uint16_t* lm_head_w,
                   const uint16_t* x, const uint16_t* res, uint16_t* kv_pages,
                   const int32_t* block_table, const int32_t* positions,
                   uint16_t* out, float* logits, int32_t* ids,
                   or_layer_trace* trace_last) {
  const int H = c->hidden, M = c->num_requests * c->tokens_per_request;
  size_t n = (size_t)M * H;
  uint16_t* xa = (uint16_t*)malloc(sizeof(uint16_t) * n);
  uint16_t* ra = (uint16_t*)malloc(sizeof(uint16_t) * n);
  uint16_t* xb = (uint16_t*)malloc(sizeof(uint16_t) * n);
  uint16_t* rb = (uint16_t*)malloc(sizeof(uint16_t) * n);
  int rc = 0;
  memcpy(xa, x, sizeof(uint16_t) * n);
  memcpy(ra, res, sizeof(uint16_t) * n);
  for (int l = 0; l < c->n_layers && rc == 0; ++l) {
    rc = or_decode_layer(c, l, &layers[l], xa, ra, kv_pages, block_table, positions, xb, rb,
                         l == c->n_layers - 1 ? trace_last : NULL);
    uint16_t* s;
    s = xa; xa = xb; xb = s;
    s = ra; ra = rb; rb = s;
  }
  if (rc == 0) {
    if (c->vocab > 0) {
      /* final residual add + RMSNorm, lm_head, greedy argmax */
      uint16_t* hfin = (uint16_t*)malloc(sizeof(uint16_t) * n);
      double* a = (double*)malloc(sizeof(double) * n);
      double* lg = (double*)malloc(sizeof(double) * (size_t)M * c->vocab);
      or_add_rmsnorm(M, H, xa, ra, final_norm_w, c->eps, rb, hfin, NULL);
      bf16_to_double_array(n, hfin, a);
      or_gemm_bf16(M, c->vocab, H, a, lm_head_w, lg);
      for (int m = 0; m < M; ++m) {
        for (int v = 0; v < c->vocab; ++v)
          logits[(size_t)m * c->vocab + v] = (float)lg[(size_t)m * c->vocab + v];
        ids[m] = or_argmax(c->vocab, logits + (size_t)m * c->vocab);
      }
      free(hfin);
      free(a);
      free(lg);
    } else {
      memcpy(out, xa, sizeof(uint16_t) * n);
      memcpy(out + n, ra, sizeof(uint16_t) * n);
    }
  }
  free(xa); free(ra); free(xb); free(rb);
  return rc;
}

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void or_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
