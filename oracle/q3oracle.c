/*
 * q3oracle.c -- plain, slow CPU reference ("the oracle") of one Qwen3-TTS-style
 * acoustic frame decode: Talker step + 15 CodePredictor steps + sampling.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant generator with the CUDA library; both sides read the same
 * weight bytes and the same uniforms, nothing else.
 *
 * Arithmetic: every model quantity is computed in double precision from the
 * stored weights (fp32 or bf16, widened exactly).  The sampler is the one
 * place where floating point decides an integer, so it runs in float with a
 * spelled-out operation order (see q3o_sample) that the CUDA sampler follows
 * independently; q3o_sample_f64 is the same rule in double, for checking.
 *
 * Sources (page title, section):
 *   [R9700]  "Running Qwen3-TTS on an AMD R9700", section "Running Qwen3-TTS":
 *            a frame is 16 codebook tokens [semantic, acoustic 1..15]; the
 *            Talker makes the semantic token, the CodePredictor fills in the
 *            15 acoustic tokens of the same frame one at a time; per-frame cost
 *            is one Talker pass plus 15 CodePredictor passes.
 *   [HIP]    "qwen3-tts-hip" README, section "Library Usage": GenerateOptions
 *            (do_sample, top_k, top_p, temperature, repetition_penalty and the
 *            subtalker_* controls), max_cache_steps; section "Python Parity
 *            Fixtures": CodePredictor token and embedding-sum parity.
 *   The workload definitions: Qwen3-style decoder layers (RMSNorm eps 1e-6,
 *   RoPE theta 1e6, GQA, SwiGLU FFN), next Talker input = sum of the previous
 *   frame's 16 code embeddings, prompt = random hidden vectors.
 *
 * Readings where the pages are silent (each restated at its use):
 *   Qwen3 per-head q/k RMSNorm before RoPE; rotate-half RoPE with
 *   inv_freq_i = theta^(-2i/hd); attention scale 1/sqrt(hd), causal, no bias,
 *   q head h reads kv head h / (Hq/Hkv); CodePredictor embeddings are
 *   Talker-width with a bias-free projection to the CodePredictor width when
 *   the widths differ; CodePredictor pass 0 carries two tokens (the Talker's
 *   final-normed hidden and the semantic code's embedding); the repetition
 *   penalty follows the usual divide-positive / multiply-negative rule over
 *   the semantic codes already emitted in the stream.
 *
 * Pins: every function here is checked by CPU tests against something other
 * than itself -- library routines (rms_norm, scaled_dot_product_attention,
 * silu, linear, torch's bf16 and float8_e4m3fn conversions), closed forms (RoPE
 * on basis vectors, one-position attention, identity-stack frames), invariants
 * (incremental decode = one causal pass), an exhaustive sampler check on a
 * fine grid of u, and the pages' frame constants and module sizes.  No
 * function is left without a pin.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q3O_NCB 16

typedef struct {
  int talker_layers, talker_hidden, talker_ffn;
  int cp_layers, cp_hidden, cp_ffn;
  int n_q_heads, n_kv_heads, head_dim;
  int codec_vocab, cp_vocab, n_codebooks;
  int kv_cap, weight_dtype, n_streams, qk_norm;
  int kv_bf16; /* Talker cache stored in bf16 (the serving configuration) */
  double rms_eps, rope_theta;
} q3o_config;

/* Per-layer pointer order: w_qkv, w_o, w_gateup, w_down,
 * g_attn_norm, g_ffn_norm, g_q_norm, g_k_norm, then the per-row scales of the
 * four matrices (FP8 weights; NULL otherwise). */
enum { L_QKV = 0, L_O, L_GU, L_DOWN, L_GATTN, L_GFFN, L_GQ, L_GK, L_SQKV, L_SO, L_SGU, L_SDOWN, L_NPTR };

/* weight_dtype: 0 fp32, 1 bf16, 2 FP8 E4M3 matrices with per-row fp32 scales
 * (gains and embedding tables then bf16). */
#define Q3O_FP8 2

typedef struct {
  const void* const* talker_layers; /* [talker_layers * L_NPTR] */
  const void* talker_g_final;
  const void* talker_w_head;        /* [V_t, D_t] */
  const void* talker_e_codec;       /* [V_t, D_t] */
  const void* const* cp_layers;     /* [cp_layers * L_NPTR] */
  const void* cp_g_final;
  const void* cp_heads;             /* [15, V_c, D_c] */
  const void* cp_embeds;            /* [15, V_c, D_t] */
  const void* cp_w_proj;            /* [D_c, D_t] or NULL */
  const float* s_head;              /* FP8: scales of talker_w_head [V_t] */
  const float* s_cp_heads;          /* FP8: [15, V_c] */
  const float* s_cp_proj;           /* FP8: [D_c] or NULL */
} q3o_weights;

typedef struct {
  int do_sample, top_k;
  float top_p, temperature, repetition_penalty;
  int sub_do_sample, sub_top_k;
  float sub_top_p, sub_temperature;
  int eos_token;     /* semantic code that ends the stream; < 0: none */
  int special_from;  /* semantic codes >= this, except eos_token, are never drawn; <= 0: none */
} q3o_sampling;

typedef struct {
  double* k; /* [layers][cap][Hkv][hd] */
  double* v;
  int bf16; /* entries hold bf16 values */
} kvbuf;

/* The bf16 value of x as a cache written from fp32 activations holds it: x
 * rounded to fp32, then to the nearest bf16 (ties to even). */
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) != 0x7f800000u) u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;
  memcpy(&f, &u, 4);
  return (double)f;
}

typedef struct {
  kvbuf talker_kv;
  int len;                 /* Talker positions filled */
  double* pending_h;       /* [D_t] final-normed hidden of the last position */
  double* pending_logits;  /* [V_t] */
  unsigned char* history;  /* [V_t] semantic codes emitted so far */
  int finished;            /* the stream fed its end-of-stream code */
} stream_state;

typedef struct {
  q3o_config c;
  q3o_weights w;
  stream_state* st;
  kvbuf cp_kv;             /* [cp_layers][16][Hkv][hd] */
} q3o_model;

/* ---------------------------------------------------------------- helpers */

/* The value of an FP8 E4M3 code: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); the all-ones code
 * (exponent 15, mantissa 7) is NaN; there are no infinities, so the largest
 * finite value is 1.75 * 2^8 = 448. */
double q3o_fp8_value(unsigned code) {
  const int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sgn ? -v : v;
}

/* Element i of a weight tensor of dtype dt (an FP8 code's value, unscaled). */
static double wval(const void* w, int dt, size_t i) {
  if (dt == 0) return (double)((const float*)w)[i];
  if (dt == Q3O_FP8) return q3o_fp8_value(((const uint8_t*)w)[i]);
  uint32_t bits = (uint32_t)((const uint16_t*)w)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* dtype of the gains and embedding tables of a model whose matrices are dt */
static int gain_dt(int dt) { return dt == Q3O_FP8 ? 1 : dt; }

/* bytes of one matrix element */
static size_t mat_esz(int dt) { return dt == 0 ? 4 : (dt == Q3O_FP8 ? 1 : 2); }

/* y[t][r] = sum_k W[r][k] x[t][k]  (W row-major [rows, cols]; FP8 rows are
 * their codes' values times the row's scale sc[r]); a plain matrix product,
 * each row widened once and then used for every token (the sums run over k in
 * order for each (t, r), whatever the number of tokens). */
static void linear(const void* W, int dt, const float* sc, int rows, int cols, const double* x, int T,
                   double* y) {
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)cols);
#pragma omp for schedule(static)
    for (int r = 0; r < rows; ++r) {
      const double srow = dt == Q3O_FP8 ? (double)sc[r] : 1.0;
      for (int k = 0; k < cols; ++k) w[k] = wval(W, dt, (size_t)r * cols + k) * srow;
      for (int t = 0; t < T; ++t) {
        double acc = 0.0;
        for (int k = 0; k < cols; ++k) acc += w[k] * x[(size_t)t * cols + k];
        y[(size_t)t * rows + r] = acc;
      }
    }
    free(w);
  }
}

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g. */
static void rmsnorm_w(const double* x, int n, const void* g, int dt, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * wval(g, dt, i);
}

/* Rotate-half RoPE at absolute position pos: pairs (i, i + hd/2) are rotated by
 * pos * theta^(-2i/hd). */
static void rope(double* v, int hd, int pos, double theta) {
  int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * i / hd);
    double a = pos * inv_freq;
    double c = cos(a), s = sin(a);
    double x0 = v[i], x1 = v[i + half];
    v[i] = x0 * c - x1 * s;
    v[i + half] = x1 * c + x0 * s;
  }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Single-query attention of Hq heads over S cached positions (GQA: q head h
 * reads kv head h / (Hq/Hkv)); max-subtracted softmax; scale 1/sqrt(hd).
 * K, V laid out [S][Hkv][hd]. */
static void attention(const double* q, const double* K, const double* V, int S, int Hq, int Hkv,
                      int hd, double* o) {
  int rep = Hq / Hkv;
  double* sc = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
  double scale = 1.0 / sqrt((double)hd);
  for (int h = 0; h < Hq; ++h) {
    int g = h / rep;
    double mx = -INFINITY;
    for (int s = 0; s < S; ++s) {
      double d = 0.0;
      for (int i = 0; i < hd; ++i) d += q[h * hd + i] * K[((size_t)s * Hkv + g) * hd + i];
      sc[s] = d * scale;
      if (sc[s] > mx) mx = sc[s];
    }
    double z = 0.0;
    for (int s = 0; s < S; ++s) {
      sc[s] = exp(sc[s] - mx);
      z += sc[s];
    }
    for (int i = 0; i < hd; ++i) {
      double acc = 0.0;
      for (int s = 0; s < S; ++s) acc += sc[s] * V[((size_t)s * Hkv + g) * hd + i];
      o[h * hd + i] = acc / z;
    }
  }
  free(sc);
}

/* --------------------------------------------------------- decoder stack */

typedef struct {
  int layers, hidden, ffn;
  const void* const* lw;
  kvbuf* kv;
  int cap;
} stack_desc;

/* Runs T consecutive tokens x[T][hidden] (positions pos0..pos0+T-1) through all
 * layers of a Qwen3-style decoder, appending each token's k, v to the cache.
 * Per layer (pre-norm):
 *   n  = RMSNorm(x);  [q; k; v] = W_qkv n
 *   q_h = RoPE(RMSNorm_hd(q_h) * g_q), k_g = RoPE(RMSNorm_hd(k_g) * g_k)
 *   x += W_o Attn(q, K[0..p], V[0..p])
 *   n' = RMSNorm(x);  x += W_down(silu(W_gate n') * (W_up n')) */
static void stack_forward(const q3o_model* m, const stack_desc* sd, double* x, int T, int pos0) {
  const q3o_config* c = &m->c;
  int D = sd->hidden, F = sd->ffn, Hq = c->n_q_heads, Hkv = c->n_kv_heads, hd = c->head_dim;
  int dt = c->weight_dtype, gdt = gain_dt(dt);
  int qkv_rows = (Hq + 2 * Hkv) * hd;
  double* n = (double*)malloc(sizeof(double) * (size_t)T * D);
  double* qkv = (double*)malloc(sizeof(double) * (size_t)T * qkv_rows);
  double* o = (double*)malloc(sizeof(double) * (size_t)T * Hq * hd);
  double* y = (double*)malloc(sizeof(double) * (size_t)T * (D > 2 * F ? D : 2 * F));
  double* a = (double*)malloc(sizeof(double) * (size_t)T * F);
  size_t layer_stride = (size_t)sd->cap * Hkv * hd;
  for (int l = 0; l < sd->layers; ++l) {
    const void* const* w = sd->lw + (size_t)l * L_NPTR;
    double* Kc = sd->kv->k + l * layer_stride;
    double* Vc = sd->kv->v + l * layer_stride;
    for (int t = 0; t < T; ++t) rmsnorm_w(x + (size_t)t * D, D, w[L_GATTN], gdt, c->rms_eps, n + (size_t)t * D);
    linear(w[L_QKV], dt, (const float*)w[L_SQKV], qkv_rows, D, n, T, qkv);
    for (int t = 0; t < T; ++t) {
      double* row = qkv + (size_t)t * qkv_rows;
      int pos = pos0 + t;
      for (int h = 0; h < Hq; ++h) {
        double* qh = row + h * hd;
        if (c->qk_norm) rmsnorm_w(qh, hd, w[L_GQ], gdt, c->rms_eps, qh);
        rope(qh, hd, pos, c->rope_theta);
      }
      for (int g = 0; g < Hkv; ++g) {
        double* kg = row + (Hq + g) * hd;
        double* vg = row + (Hq + Hkv + g) * hd;
        if (c->qk_norm) rmsnorm_w(kg, hd, w[L_GK], gdt, c->rms_eps, kg);
        rope(kg, hd, pos, c->rope_theta);
        double* kc = Kc + ((size_t)pos * Hkv + g) * hd;
        double* vc = Vc + ((size_t)pos * Hkv + g) * hd;
        for (int i = 0; i < hd; ++i) {
          kc[i] = sd->kv->bf16 ? round_bf16(kg[i]) : kg[i];
          vc[i] = sd->kv->bf16 ? round_bf16(vg[i]) : vg[i];
        }
      }
    }
    /* causal: token t sees positions 0..pos0+t, itself included (tokens are
     * independent here: each reads the cache filled above) */
#pragma omp parallel for schedule(dynamic, 4)
    for (int t = 0; t < T; ++t)
      attention(qkv + (size_t)t * qkv_rows, Kc, Vc, pos0 + t + 1, Hq, Hkv, hd, o + (size_t)t * Hq * hd);
    linear(w[L_O], dt, (const float*)w[L_SO], D, Hq * hd, o, T, y);
    for (size_t i = 0; i < (size_t)T * D; ++i) x[i] += y[i];
    for (int t = 0; t < T; ++t) rmsnorm_w(x + (size_t)t * D, D, w[L_GFFN], gdt, c->rms_eps, n + (size_t)t * D);
    linear(w[L_GU], dt, (const float*)w[L_SGU], 2 * F, D, n, T, y);
    for (int t = 0; t < T; ++t)
      for (int f = 0; f < F; ++f)
        a[(size_t)t * F + f] = silu(y[(size_t)t * 2 * F + f]) * y[(size_t)t * 2 * F + F + f];
    linear(w[L_DOWN], dt, (const float*)w[L_SDOWN], D, F, a, T, y);
    for (size_t i = 0; i < (size_t)T * D; ++i) x[i] += y[i];
  }
  free(n); free(qkv); free(o); free(y); free(a);
}

/* ----------------------------------------------------------- the sampler */

/* exp for x <= 0 in float, written from the Cody-Waite method (W. J. Cody and
 * W. Waite, "Software Manual for the Elementary Functions", 1980): k = rint(x /
 * ln 2), r = x - k ln 2 with ln 2 split in two parts so k * hi is exact, then a
 * degree-7 Taylor polynomial of e^r in Horner form with explicit fused
 * multiply-adds, scaled by 2^k.  Inputs below -80 give 0. */
float q3o_expf(float x) {
  if (!(x >= -80.0f)) return 0.0f;
  float kf = rintf(x * 1.44269504088896341f);
  float r = fmaf(-kf, 0.693145751953125f, x);
  r = fmaf(-kf, 1.42860682030941723212e-6f, r);
  float p = 1.98412698412698413e-4f;
  p = fmaf(p, r, 1.38888888888888889e-3f);
  p = fmaf(p, r, 8.33333333333333333e-3f);
  p = fmaf(p, r, 4.16666666666666667e-2f);
  p = fmaf(p, r, 1.66666666666666667e-1f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  return ldexpf(p, (int)kf);
}

typedef struct { float v; int i; } cand;

static int cand_cmp(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

/* Whether id may be drawn: ids >= special_from (when special_from > 0) are
 * special codes, of which only eos_token may be drawn. */
static int allowed_id(int id, int special_from, int eos_token) {
  return special_from <= 0 || id < special_from || id == eos_token;
}

/* The token rule, in float, in this order ("qwen3-tts-hip" README, "Library
 * Usage": repetition_penalty, temperature, top_k, top_p, do_sample; the
 * candidate set first drops the special codes that may not be drawn):
 *  0. candidates: the ids allowed_id() admits (V_eff of them);
 *  1. repetition penalty rho != 1: for each id in the history,
 *     l = l > 0 ? l / rho : l * rho;
 *  2. greedy (do_sample == 0): the largest l, lowest index on ties;
 *  3. l = l / T for every id;
 *  4. order ids by (l descending, index ascending); keep the first k
 *     (k <= 0 or k >= V_eff keeps all V_eff);
 *  5. m = first kept l; w_i = q3o_expf(l_i - m) in that order;
 *  6. top-p < 1: Z = w_0 + w_1 + ... (left to right, float); keep the shortest
 *     prefix whose running sum reaches top_p * Z (>=);
 *  7. Z = running float sum of the kept w; t = u * Z; the pick is the first
 *     kept id whose running sum is > t, else the last kept id. */
int q3o_sample(const float* logits, int V, int do_sample, int top_k, float top_p, float temperature,
               float rep_penalty, const unsigned char* history, float u, int special_from, int eos_token) {
  float* l = (float*)malloc(sizeof(float) * (size_t)V);
  memcpy(l, logits, sizeof(float) * (size_t)V);
  if (history && rep_penalty != 1.0f)
    for (int i = 0; i < V; ++i)
      if (history[i]) l[i] = l[i] > 0.0f ? l[i] / rep_penalty : l[i] * rep_penalty;
  if (!do_sample) {
    int best = -1;
    for (int i = 0; i < V; ++i)
      if (allowed_id(i, special_from, eos_token) && (best < 0 || l[i] > l[best])) best = i;
    free(l);
    return best;
  }
  cand* cs = (cand*)malloc(sizeof(cand) * (size_t)V);
  int Ve = 0;
  for (int i = 0; i < V; ++i) {
    if (!allowed_id(i, special_from, eos_token)) continue;
    cs[Ve].v = l[i] / temperature;
    cs[Ve].i = i;
    ++Ve;
  }
  qsort(cs, (size_t)Ve, sizeof(cand), cand_cmp);
  int K = (top_k <= 0 || top_k >= Ve) ? Ve : top_k;
  float m = cs[0].v;
  float* w = (float*)malloc(sizeof(float) * (size_t)K);
  for (int i = 0; i < K; ++i) w[i] = q3o_expf(cs[i].v - m);
  if (top_p < 1.0f) {
    float z = 0.0f;
    for (int i = 0; i < K; ++i) z = z + w[i];
    float tp = top_p * z, run = 0.0f;
    for (int i = 0; i < K; ++i) {
      run = run + w[i];
      if (run >= tp) { K = i + 1; break; }
    }
  }
  float z = 0.0f;
  for (int i = 0; i < K; ++i) z = z + w[i];
  float t = u * z, run = 0.0f;
  int pick = cs[K - 1].i;
  for (int i = 0; i < K; ++i) {
    run = run + w[i];
    if (run > t) { pick = cs[i].i; break; }
  }
  free(w); free(cs); free(l);
  return pick;
}

typedef struct { double v; int i; } candd;

static int candd_cmp(const void* a, const void* b) {
  const candd* x = (const candd*)a;
  const candd* y = (const candd*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i > y->i) - (x->i < y->i);
}

/* The same rule in double with libm exp (a check of q3o_sample: the two may
 * differ only where u * Z lands within rounding of a CDF boundary).  *margin
 * receives |running_sum - u*Z| / Z at the nearest boundary. */
int q3o_sample_f64(const float* logits, int V, int do_sample, int top_k, double top_p,
                   double temperature, double rep_penalty, const unsigned char* history, double u,
                   double* margin, int special_from, int eos_token) {
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  for (int i = 0; i < V; ++i) l[i] = logits[i];
  if (history && rep_penalty != 1.0)
    for (int i = 0; i < V; ++i)
      if (history[i]) l[i] = l[i] > 0.0 ? l[i] / rep_penalty : l[i] * rep_penalty;
  if (!do_sample) {
    int best = -1;
    for (int i = 0; i < V; ++i)
      if (allowed_id(i, special_from, eos_token) && (best < 0 || l[i] > l[best])) best = i;
    if (margin) *margin = INFINITY;
    free(l);
    return best;
  }
  candd* cs = (candd*)malloc(sizeof(candd) * (size_t)V);
  int Ve = 0;
  for (int i = 0; i < V; ++i) {
    if (!allowed_id(i, special_from, eos_token)) continue;
    cs[Ve].v = l[i] / temperature;
    cs[Ve].i = i;
    ++Ve;
  }
  qsort(cs, (size_t)Ve, sizeof(candd), candd_cmp);
  int K = (top_k <= 0 || top_k >= Ve) ? Ve : top_k;
  double* w = (double*)malloc(sizeof(double) * (size_t)K);
  for (int i = 0; i < K; ++i) w[i] = exp(cs[i].v - cs[0].v);
  if (top_p < 1.0) {
    double z = 0.0;
    for (int i = 0; i < K; ++i) z += w[i];
    double run = 0.0;
    for (int i = 0; i < K; ++i) {
      run += w[i];
      if (run >= top_p * z) { K = i + 1; break; }
    }
  }
  double z = 0.0;
  for (int i = 0; i < K; ++i) z += w[i];
  double t = u * z, run = 0.0, best_margin = INFINITY;
  int pick = cs[K - 1].i, found = 0;
  for (int i = 0; i < K; ++i) {
    run += w[i];
    double d = fabs(run - t) / z;
    if (d < best_margin) best_margin = d;
    if (!found && run > t) { pick = cs[i].i; found = 1; }
  }
  if (margin) *margin = best_margin;
  free(w); free(cs); free(l);
  return pick;
}

/* ------------------------------------------------------------- the model */

static void talker_stack(const q3o_model* m, stream_state* st, stack_desc* sd) {
  sd->layers = m->c.talker_layers;
  sd->hidden = m->c.talker_hidden;
  sd->ffn = m->c.talker_ffn;
  sd->lw = m->w.talker_layers;
  sd->kv = &st->talker_kv;
  sd->cap = m->c.kv_cap;
}

static void cp_stack(q3o_model* m, stack_desc* sd) {
  sd->layers = m->c.cp_layers;
  sd->hidden = m->c.cp_hidden;
  sd->ffn = m->c.cp_ffn;
  sd->lw = m->w.cp_layers;
  sd->kv = &m->cp_kv;
  sd->cap = m->c.n_codebooks;
}

/* Final norm + codec head of the Talker at the last of T tokens: the pending
 * state from which the next frame's semantic token is drawn. */
static void talker_pending(q3o_model* m, stream_state* st, const double* x_last) {
  const q3o_config* c = &m->c;
  rmsnorm_w(x_last, c->talker_hidden, m->w.talker_g_final, gain_dt(c->weight_dtype), c->rms_eps, st->pending_h);
  linear(m->w.talker_w_head, c->weight_dtype, m->w.s_head, c->codec_vocab, c->talker_hidden, st->pending_h, 1,
         st->pending_logits);
}

void* q3o_create(const q3o_config* cfg, const q3o_weights* w) {
  q3o_model* m = (q3o_model*)calloc(1, sizeof(q3o_model));
  m->c = *cfg;
  m->w = *w;
  const q3o_config* c = &m->c;
  size_t kv = (size_t)c->talker_layers * c->kv_cap * c->n_kv_heads * c->head_dim;
  m->st = (stream_state*)calloc((size_t)c->n_streams, sizeof(stream_state));
  for (int s = 0; s < c->n_streams; ++s) {
    m->st[s].talker_kv.bf16 = c->kv_bf16;
    m->st[s].talker_kv.k = (double*)calloc(kv, sizeof(double));
    m->st[s].talker_kv.v = (double*)calloc(kv, sizeof(double));
    m->st[s].pending_h = (double*)calloc((size_t)c->talker_hidden, sizeof(double));
    m->st[s].pending_logits = (double*)calloc((size_t)c->codec_vocab, sizeof(double));
    m->st[s].history = (unsigned char*)calloc((size_t)c->codec_vocab, 1);
  }
  size_t ckv = (size_t)c->cp_layers * c->n_codebooks * c->n_kv_heads * c->head_dim;
  m->cp_kv.k = (double*)calloc(ckv, sizeof(double));
  m->cp_kv.v = (double*)calloc(ckv, sizeof(double));
  return m;
}

void q3o_destroy(void* h) {
  q3o_model* m = (q3o_model*)h;
  if (!m) return;
  for (int s = 0; s < m->c.n_streams; ++s) {
    free(m->st[s].talker_kv.k); free(m->st[s].talker_kv.v);
    free(m->st[s].pending_h); free(m->st[s].pending_logits); free(m->st[s].history);
  }
  free(m->st); free(m->cp_kv.k); free(m->cp_kv.v); free(m);
}

int q3o_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Thread count of later parallel regions (timing on a given number of cores). */
void q3o_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Prompt (N(0,1) hidden vectors used directly as Talker inputs) at positions
 * 0..len-1; the stream restarts.  Returns 0, or -1 if len is out of range. */
int q3o_prefill(void* h, int stream, const float* embeds, int len) {
  q3o_model* m = (q3o_model*)h;
  const q3o_config* c = &m->c;
  if (stream < 0 || stream >= c->n_streams || len < 1 || len >= c->kv_cap) return -1;
  stream_state* st = &m->st[stream];
  memset(st->history, 0, (size_t)c->codec_vocab);
  st->finished = 0;
  int D = c->talker_hidden;
  double* x = (double*)malloc(sizeof(double) * (size_t)len * D);
  for (size_t i = 0; i < (size_t)len * D; ++i) x[i] = embeds[i];
  stack_desc sd;
  talker_stack(m, st, &sd);
  stack_forward(m, &sd, x, len, 0);
  st->len = len;
  talker_pending(m, st, x + (size_t)(len - 1) * D);
  free(x);
  return 0;
}

/* Copies the pending Talker state (final-normed hidden [D_t], logits [V_t]). */
void q3o_pending(void* h, int stream, double* hidden, double* logits) {
  q3o_model* m = (q3o_model*)h;
  stream_state* st = &m->st[stream];
  if (hidden) memcpy(hidden, st->pending_h, sizeof(double) * (size_t)m->c.talker_hidden);
  if (logits) memcpy(logits, st->pending_logits, sizeof(double) * (size_t)m->c.codec_vocab);
}

int q3o_length(void* h, int stream) { return ((q3o_model*)h)->st[stream].len; }

/* CodePredictor pass: tokens u[T][D_t] (projected to D_c when the widths
 * differ) at CodePredictor positions pos0.., then the final norm and head
 * `head` at the last token.  logits: [V_c] in double. */
static void cp_pass(q3o_model* m, const double* u, int T, int pos0, int head, double* logits) {
  const q3o_config* c = &m->c;
  int Dt = c->talker_hidden, Dc = c->cp_hidden, dt = c->weight_dtype;
  double* z = (double*)malloc(sizeof(double) * (size_t)T * Dc);
  if (c->talker_hidden != c->cp_hidden)
    linear(m->w.cp_w_proj, dt, m->w.s_cp_proj, Dc, Dt, u, T, z);
  else
    memcpy(z, u, sizeof(double) * (size_t)T * Dc);
  stack_desc sd;
  cp_stack(m, &sd);
  stack_forward(m, &sd, z, T, pos0);
  double* hn = (double*)malloc(sizeof(double) * (size_t)Dc);
  rmsnorm_w(z + (size_t)(T - 1) * Dc, Dc, m->w.cp_g_final, gain_dt(dt), c->rms_eps, hn);
  const void* W = (const char*)m->w.cp_heads + (size_t)head * c->cp_vocab * Dc * mat_esz(dt);
  linear(W, dt, m->w.s_cp_heads ? m->w.s_cp_heads + (size_t)head * c->cp_vocab : NULL, c->cp_vocab, Dc, hn, 1,
         logits);
  free(hn); free(z);
}

static void embed_row(const q3o_model* m, const void* table, size_t row, double* out) {
  int Dt = m->c.talker_hidden;
  for (int i = 0; i < Dt; ++i) out[i] = wval(table, gain_dt(m->c.weight_dtype), row * Dt + i);
}

/* One acoustic frame of one stream ([R9700] "Running Qwen3-TTS"):
 *   c0 from the pending Talker logits (semantic rule, history, u[0]);
 *   CodePredictor pass 0 on [h_T, E_t[c0]] at positions 0, 1 -> head 0 -> c1;
 *   pass j = 1..14 on E_cp[j-1][c_j] at position j+1 -> head j -> c_{j+1};
 *   x = E_t[c0] + sum_{j=1..15} E_cp[j-1][c_j] (the embedding sum);
 *   one Talker step at the next position -> new pending state.
 * codes_out[16] gets the drawn codes.  If forced (16 codes) is given, the
 * forced codes are fed forward instead of the drawn ones (teacher forcing).
 * logits_out (optional, float [V_t + 15 V_c]) receives the raw logits behind
 * each draw.  Returns 0, or -1 when the Talker cache is full. */
int q3o_step_frame(void* h, int stream, const q3o_sampling* sp, const float* u, const int* forced,
                   int* codes_out, float* logits_out) {
  q3o_model* m = (q3o_model*)h;
  const q3o_config* c = &m->c;
  stream_state* st = &m->st[stream];
  if (st->len >= c->kv_cap) return -1;
  int Dt = c->talker_hidden, Vt = c->codec_vocab, Vc = c->cp_vocab, dt = gain_dt(c->weight_dtype);
  size_t esz = dt == 0 ? 4 : 2; /* embedding tables */
  int fed[Q3O_NCB];
  float* lf = (float*)malloc(sizeof(float) * (size_t)(Vt > Vc ? Vt : Vc));
  double* ld = (double*)malloc(sizeof(double) * (size_t)Vc);

  /* a finished stream yields no codes and keeps its state */
  if (st->finished) {
    for (int j = 0; j < c->n_codebooks; ++j) codes_out[j] = -1;
    free(lf); free(ld);
    return 0;
  }
  for (int i = 0; i < Vt; ++i) lf[i] = (float)st->pending_logits[i];
  if (logits_out) memcpy(logits_out, lf, sizeof(float) * (size_t)Vt);
  codes_out[0] = q3o_sample(lf, Vt, sp->do_sample, sp->top_k, sp->top_p, sp->temperature,
                            sp->repetition_penalty, st->history, u[0], sp->special_from, sp->eos_token);
  fed[0] = forced ? forced[0] : codes_out[0];
  /* the end-of-stream code ends the stream with this frame: no acoustic
   * codes, no Talker step */
  if (sp->eos_token >= 0 && fed[0] == sp->eos_token) {
    st->finished = 1;
    for (int j = 1; j < c->n_codebooks; ++j) codes_out[j] = -1;
    free(lf); free(ld);
    return 0;
  }
  st->history[fed[0]] = 1;

  /* CodePredictor: the cache restarts every frame */
  double* tok = (double*)malloc(sizeof(double) * (size_t)2 * Dt);
  memcpy(tok, st->pending_h, sizeof(double) * (size_t)Dt);
  embed_row(m, m->w.talker_e_codec, (size_t)fed[0], tok + Dt);
  for (int j = 0; j < c->n_codebooks - 1; ++j) {
    if (j == 0) {
      cp_pass(m, tok, 2, 0, 0, ld);
    } else {
      const void* E = (const char*)m->w.cp_embeds + (size_t)(j - 1) * Vc * Dt * esz;
      embed_row(m, E, (size_t)fed[j], tok);
      cp_pass(m, tok, 1, j + 1, j, ld);
    }
    for (int i = 0; i < Vc; ++i) lf[i] = (float)ld[i];
    if (logits_out) memcpy(logits_out + Vt + (size_t)j * Vc, lf, sizeof(float) * (size_t)Vc);
    codes_out[j + 1] = q3o_sample(lf, Vc, sp->sub_do_sample, sp->sub_top_k, sp->sub_top_p,
                                  sp->sub_temperature, 1.0f, NULL, u[j + 1], 0, -1);
    fed[j + 1] = forced ? forced[j + 1] : codes_out[j + 1];
  }

  /* next Talker input: sum of the frame's 16 code embeddings */
  double* x = (double*)calloc((size_t)Dt, sizeof(double));
  embed_row(m, m->w.talker_e_codec, (size_t)fed[0], tok);
  for (int i = 0; i < Dt; ++i) x[i] += tok[i];
  for (int j = 1; j < c->n_codebooks; ++j) {
    const void* E = (const char*)m->w.cp_embeds + (size_t)(j - 1) * Vc * Dt * esz;
    embed_row(m, E, (size_t)fed[j], tok);
    for (int i = 0; i < Dt; ++i) x[i] += tok[i];
  }
  stack_desc sd;
  talker_stack(m, st, &sd);
  stack_forward(m, &sd, x, 1, st->len);
  st->len += 1;
  talker_pending(m, st, x);
  free(x); free(tok); free(ld); free(lf);
  return 0;
}

/* ----------------------------------------- small pieces for the pin tests */

void q3o_rmsnorm(const double* x, int n, const float* g, double eps, double* y) {
  rmsnorm_w(x, n, g, 0, eps, y);
}

void q3o_rope(double* v, int hd, int pos, double theta) { rope(v, hd, pos, theta); }

void q3o_attention(const double* q, const double* K, const double* V, int S, int Hq, int Hkv, int hd,
                   double* o) {
  attention(q, K, V, S, Hq, Hkv, hd, o);
}

/* Runs T tokens through the Talker stack of stream 0 starting at pos0 and
 * returns the stack output x (pre final norm), for layer-level pins. */
void q3o_talker_stack(void* h, int stream, double* x, int T, int pos0) {
  q3o_model* m = (q3o_model*)h;
  stack_desc sd;
  talker_stack(m, &m->st[stream], &sd);
  stack_forward(m, &sd, x, T, pos0);
}

/* The frame's whole CodePredictor sequence in one causal pass, for the
 * incremental-cache pin: tokens [16][D_t] = [h_T, E_t[c0], E_cp[0][c1], ...,
 * E_cp[13][c14]] at positions 0..15; head j is applied at position j+1.
 * logits: float [15][V_c]. */
void q3o_cp_full(void* h, const double* tokens, float* logits) {
  q3o_model* m = (q3o_model*)h;
  const q3o_config* c = &m->c;
  int T = c->n_codebooks, Dt = c->talker_hidden, Dc = c->cp_hidden, Vc = c->cp_vocab;
  int dt = c->weight_dtype;
  double* z = (double*)malloc(sizeof(double) * (size_t)T * Dc);
  if (Dt != Dc)
    linear(m->w.cp_w_proj, dt, m->w.s_cp_proj, Dc, Dt, tokens, T, z);
  else
    memcpy(z, tokens, sizeof(double) * (size_t)T * Dc);
  stack_desc sd;
  cp_stack(m, &sd);
  stack_forward(m, &sd, z, T, 0);
  double* hn = (double*)malloc(sizeof(double) * (size_t)Dc);
  double* ld = (double*)malloc(sizeof(double) * (size_t)Vc);
  for (int j = 0; j < T - 1; ++j) {
    rmsnorm_w(z + (size_t)(j + 1) * Dc, Dc, m->w.cp_g_final, gain_dt(dt), c->rms_eps, hn);
    const void* W = (const char*)m->w.cp_heads + (size_t)j * Vc * Dc * mat_esz(dt);
    linear(W, dt, m->w.s_cp_heads ? m->w.s_cp_heads + (size_t)j * Vc : NULL, Vc, Dc, hn, 1, ld);
    for (int i = 0; i < Vc; ++i) logits[(size_t)j * Vc + i] = (float)ld[i];
  }
  free(ld); free(hn); free(z);
}
