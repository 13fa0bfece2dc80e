/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.  A plain, slow CPU restatement of the
 * frame-locked batched decode step, used to check the CUDA library.  Only the
 * tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes follows the pages' description of the frame step:
 *   - "PersonaPlex 7B, 80 sessions, one H100" (narilabs blog), sections
 *     "What Real-time Means for a Full-duplex Agent" (one 80 ms frame per
 *     forward pass), "Compressing the Temporal KV cache" (bf16 weights and
 *     activations, FP8 temporal K/V cache) and "A server built around the
 *     conversation clock" (every session advances together, fixed shape);
 *   - the dotwave.ai case study, "02 / The solution" and "04 / Under the
 *     hood" (weights shared across sessions, state kept between beats).
 * The pages give no layer-level definition; the decoder layer (RMSNorm, QKV,
 * RoPE, FP8 K/V append, attention, output projection, SwiGLU MLP) and its
 * shapes come from the workload definition, and every point the pages leave
 * open is taken at its plainest reading (listed in the design notes):
 *   rounding to bf16 only at the projection inputs (normed x, attention
 *   output, SwiGLU output) and at y; rotate-half RoPE with pairs (i, i+D/2);
 *   softmax scale 1/sqrt(D) over slots 0..pos inclusive; no biases, no GQA,
 *   no final norm or LM head; FP8 scale amax/448 per (session, layer, K|V,
 *   head, token), quantised by fp32 division.
 * Arithmetic is fp64 everywhere except the FP8 quantiser, which is the fp32
 * definition itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int n_layers, d_model, n_heads, head_dim, ffn;
  float rms_eps, rope_base;
} oracle_cfg;

/* ------------------------------------------------------------------ bf16 */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bfloat16 (8 significant bits, ties to even),
 * straight from the double (no intermediate fp32 rounding). */
uint16_t oracle_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1) */
  int e = ex - 1;  /* a in [2^e, 2^(e+1)) */
  int ulp_e = (e < -126) ? -133 : e - 7;
  double q = ldexp(a, -ulp_e);
  double r = nearbyint(q); /* default rounding mode: to nearest, ties to even */
  double v = ldexp(r, ulp_e);
  if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)v; /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

double oracle_bf16_round(double x) { return oracle_bf16_to_double(oracle_double_to_bf16(x)); }

/* -------------------------------------------------------------- FP8 E4M3 */
/* OCP 8-bit floating point, E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa
 * bits; no infinities; S.1111.111 is NaN; largest finite magnitude 448. */
double oracle_e4m3_decode(uint8_t c) {
  int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Nearest of the 127 finite non-negative magnitudes (codes 0x00..0x7E, which
 * increase with the code), ties to the code whose last bit is 0; magnitudes at
 * or beyond 448 saturate to 448; the sign bit is kept (so -0 and negative
 * underflow give 0x80). */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E; /* largest code with decode(code) <= a */
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (oracle_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
  }
  int c = lo;
  if (c < 0x7E) {
    double d0 = a - oracle_e4m3_decode((uint8_t)c);
    double d1 = oracle_e4m3_decode((uint8_t)(c + 1)) - a;
    if (d1 < d0 || (d1 == d0 && ((c + 1) & 1) == 0)) c = c + 1;
  }
  return sign | (uint8_t)c;
}

void oracle_e4m3_encode_many(const float* v, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

/* Per-row FP8 quantiser: amax over the row, scale = amax / 448 (fp32), code =
 * E4M3(v / scale) with the division in fp32.  A zero scale gives all-zero
 * codes and a stored scale of 0. */
void oracle_quantize_row(const float* v, int D, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int i = 0; i < D; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  *scale = s;
  for (int i = 0; i < D; ++i) codes[i] = (s == 0.0f) ? 0 : oracle_e4m3_encode(v[i] / s);
}

void oracle_quantize_rows(const float* v, int64_t rows, int D, uint8_t* codes, float* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    oracle_quantize_row(v + r * D, D, codes + r * D, scales + r);
}

/* ------------------------------------------------------------ layer parts */
/* out = r / sqrt(mean(r^2) + eps) * g */
void oracle_rmsnorm(const double* r, const uint16_t* g, int d, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < d; ++i) ss += r[i] * r[i];
  double inv = 1.0 / sqrt(ss / d + eps);
  for (int i = 0; i < d; ++i) out[i] = r[i] * inv * oracle_bf16_to_double(g[i]);
}

/* y[n] = sum_k W[n][k] * x[k], W stored [N][K] in bf16. */
void oracle_matvec(const uint16_t* W, int N, int K, const double* x, double* y) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint16_t* w = W + (int64_t)n * K;
    double acc = 0.0;
    for (int k = 0; k < K; ++k) acc += oracle_bf16_to_double(w[k]) * x[k];
    y[n] = acc;
  }
}

/* Rotate-half RoPE on one head vector: pairs (i, i + D/2), angle pos * theta_i,
 * theta_i = base^(-2i/D). */
void oracle_rope(double* v, int D, int pos, double base) {
  int half = D / 2;
  for (int i = 0; i < half; ++i) {
    double theta = pow(base, -2.0 * i / D);
    double ang = (double)pos * theta;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = a * s + b * c;
  }
}

/* Attention of one head over cache slots 0..pos inclusive:
 * score_t = (q . dec(kc_t)) * ks_t / sqrt(D); p = softmax(score);
 * o = sum_t p_t * vs_t * dec(vc_t).  kc/vc are [T][D] codes, ks/vs [T]. */
void oracle_attention_head(const double* q, const uint8_t* kc, const float* ks,
                           const uint8_t* vc, const float* vs, int pos, int D, double* o) {
  int n = pos + 1;
  double* sc = (double*)malloc(sizeof(double) * (size_t)n);
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double dot = 0.0;
    for (int i = 0; i < D; ++i) dot += q[i] * oracle_e4m3_decode(kc[(int64_t)t * D + i]);
    sc[t] = dot * (double)ks[t] / sqrt((double)D);
    if (sc[t] > m) m = sc[t];
  }
  double l = 0.0;
  for (int i = 0; i < D; ++i) o[i] = 0.0;
  for (int t = 0; t < n; ++t) {
    double p = exp(sc[t] - m);
    l += p;
    double w = p * (double)vs[t];
    for (int i = 0; i < D; ++i) o[i] += w * oracle_e4m3_decode(vc[(int64_t)t * D + i]);
  }
  for (int i = 0; i < D; ++i) o[i] /= l;
  free(sc);
}

double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------- the step */
static int64_t layer_elems(const oracle_cfg* c) {
  int64_t d = c->d_model, HD = (int64_t)c->n_heads * c->head_dim, F = c->ffn;
  return d + 3 * HD * d + d * HD + d + 2 * F * d + d * F;
}

/*
 * One frame for n independent sessions.  kv is [L][2][n][H][T_max][D] codes,
 * kv_scales [L][2][n][H][T_max]; both are read at slots 0..pos[s]-1 and slot
 * pos[s] is written (then read back quantised).  x, y are [n][d] bf16.
 * A negative pos[s] marks an empty slot (a fixed-shape batch with a place
 * not taken by a session): y[s] = x[s] and its cache is not touched.
 * y_exact (nullable) receives the fp64 residual before the final rounding;
 * kv_new (nullable) receives the fp32 K/V values that were quantised,
 * [L][2][n][H][D] (NaN for empty slots).  round_acts = 0 skips the bf16
 * rounding of activations (an fp64 "pure" variant, for information).
 * Returns 0, or -(s+1) for the first session whose position is >= T_max.
 */
int oracle_step(const oracle_cfg* c, int T_max, const uint16_t* weights, int n, uint8_t* kv,
                float* kv_scales, const int32_t* pos, const uint16_t* x, uint16_t* y,
                double* y_exact, int round_acts, float* kv_new) {
  const int L = c->n_layers, d = c->d_model, H = c->n_heads, D = c->head_dim, F = c->ffn;
  const int HD = H * D;
  const int64_t le = layer_elems(c);
  for (int s = 0; s < n; ++s)
    if (pos[s] >= T_max) return -(s + 1);

  double* r = (double*)malloc(sizeof(double) * d);
  double* xn = (double*)malloc(sizeof(double) * d);
  double* qkv = (double*)malloc(sizeof(double) * 3 * HD);
  double* att = (double*)malloc(sizeof(double) * HD);
  double* tmp = (double*)malloc(sizeof(double) * (d > 2 * F ? d : 2 * F));
  double* u = (double*)malloc(sizeof(double) * F);
  float* row = (float*)malloc(sizeof(float) * D);

  for (int s = 0; s < n; ++s) {
    const int P = pos[s];
    if (P < 0) {
      /* empty slot: the session takes no part in the frame; y = x, no cache access */
      for (int i = 0; i < d; ++i) {
        y[(int64_t)s * d + i] = x[(int64_t)s * d + i];
        if (y_exact) y_exact[(int64_t)s * d + i] = oracle_bf16_to_double(x[(int64_t)s * d + i]);
      }
      if (kv_new)
        for (int l = 0; l < L; ++l)
          for (int which = 0; which < 2; ++which)
            for (int h = 0; h < H; ++h)
              for (int i = 0; i < D; ++i)
                kv_new[((((int64_t)l * 2 + which) * n + s) * H + h) * D + i] = NAN;
      continue;
    }
    for (int i = 0; i < d; ++i) r[i] = oracle_bf16_to_double(x[(int64_t)s * d + i]);
    for (int l = 0; l < L; ++l) {
      const uint16_t* Wl = weights + (int64_t)l * le;
      const uint16_t* g_attn = Wl;
      const uint16_t* wqkv = g_attn + d;
      const uint16_t* wo = wqkv + (int64_t)3 * HD * d;
      const uint16_t* g_mlp = wo + (int64_t)d * HD;
      const uint16_t* wgu = g_mlp + d;
      const uint16_t* wdown = wgu + (int64_t)2 * F * d;

      /* attention block */
      oracle_rmsnorm(r, g_attn, d, c->rms_eps, xn);
      if (round_acts) for (int i = 0; i < d; ++i) xn[i] = oracle_bf16_round(xn[i]);
      oracle_matvec(wqkv, 3 * HD, d, xn, qkv);
      double* q = qkv;
      double* k = qkv + HD;
      double* v = qkv + 2 * HD;
      for (int h = 0; h < H; ++h) {
        oracle_rope(q + h * D, D, P, c->rope_base);
        oracle_rope(k + h * D, D, P, c->rope_base);
      }
      for (int which = 0; which < 2; ++which) {
        const double* src = which ? v : k;
        for (int h = 0; h < H; ++h) {
          int64_t sh = (((int64_t)l * 2 + which) * n + s) * H + h;
          for (int i = 0; i < D; ++i) row[i] = (float)src[h * D + i];
          if (kv_new)
            memcpy(kv_new + ((((int64_t)l * 2 + which) * n + s) * H + h) * D, row, sizeof(float) * D);
          oracle_quantize_row(row, D, kv + (sh * T_max + P) * D, kv_scales + sh * T_max + P);
        }
      }
#pragma omp parallel for schedule(static)
      for (int h = 0; h < H; ++h) {
        int64_t shk = (((int64_t)l * 2 + 0) * n + s) * H + h;
        int64_t shv = (((int64_t)l * 2 + 1) * n + s) * H + h;
        oracle_attention_head(q + h * D, kv + shk * T_max * D, kv_scales + shk * T_max,
                              kv + shv * T_max * D, kv_scales + shv * T_max, P, D, att + h * D);
      }
      if (round_acts) for (int i = 0; i < HD; ++i) att[i] = oracle_bf16_round(att[i]);
      oracle_matvec(wo, d, HD, att, tmp);
      for (int i = 0; i < d; ++i) r[i] += tmp[i];

      /* MLP block */
      oracle_rmsnorm(r, g_mlp, d, c->rms_eps, xn);
      if (round_acts) for (int i = 0; i < d; ++i) xn[i] = oracle_bf16_round(xn[i]);
      oracle_matvec(wgu, 2 * F, d, xn, tmp);
      for (int i = 0; i < F; ++i) {
        u[i] = oracle_silu(tmp[i]) * tmp[F + i];
        if (round_acts) u[i] = oracle_bf16_round(u[i]);
      }
      oracle_matvec(wdown, d, F, u, tmp);
      for (int i = 0; i < d; ++i) r[i] += tmp[i];
    }
    for (int i = 0; i < d; ++i) {
      y[(int64_t)s * d + i] = oracle_double_to_bf16(r[i]);
      if (y_exact) y_exact[(int64_t)s * d + i] = r[i];
    }
  }
  free(r); free(xn); free(qkv); free(att); free(tmp); free(u); free(row);
  return 0;
}

/*
 * The projection between the dependent steps of the inner depth loop (the
 * narilabs blog, "Predictable GPU execution": the Depformer's 8-step
 * autoregressive loop per frame): x_next[s] = bf16(W_p y[s]), W_p a bf16
 * [d][d] matrix (row = output), fp64 accumulation, one rounding to bf16.
 */
void oracle_proj(const uint16_t* wp, int d, int n, const uint16_t* y, uint16_t* x_next) {
  double* a = (double*)malloc(sizeof(double) * d);
  double* o = (double*)malloc(sizeof(double) * d);
  for (int s = 0; s < n; ++s) {
    for (int i = 0; i < d; ++i) a[i] = oracle_bf16_to_double(y[(int64_t)s * d + i]);
    oracle_matvec(wp, d, d, a, o);
    for (int i = 0; i < d; ++i) x_next[(int64_t)s * d + i] = oracle_double_to_bf16(o[i]);
  }
  free(a);
  free(o);
}

/* ------------------------------------------------------------------ hybrid
 * The hybrid recurrent step (48 layers of width 4096 at full size, an
 * attention block every sixth layer, 64 state heads of 64 x 128: the
 * NemotronH-style thinker of the vllm-omni recipe page, "Summary";
 * "recurrent_state": "FP32" in the dotwave.ai profile.json).  The pages give
 * no layer definition; readings: every layer is a pre-norm residual block
 * without an MLP.  Layer l is an
 * attention block (the decoder's attention half: RMSNorm, QKV, RoPE, FP8
 * append, attention, O) when l % attn_every == attn_every - 1, else a
 * Mamba2-style selective-state block:
 *   zxbcdt = W_in xn, split [z d_i | x d_i | B N | C N | dt Hs] (one group,
 *   no conv1d); per head: dt = softplus(dt + dt_bias), A = -exp(A_log),
 *   a = exp(dt A); per head dim p and state n:
 *   h[p][n] <- a h[p][n] + dt B[n] x[p]  (stored in fp32: the state is fp32),
 *   y[p] = sum_n C[n] h[p][n] + D x[p];  out = bf16(y * silu(z));
 *   r += W_out out.
 * Blob per layer (bf16, [out][in]): Mamba: g, W_in [2 d_i + 2N + Hs][d],
 * W_out [d][d_i], A_log [Hs], dt_bias [Hs], D [Hs] (this last block padded to
 * a multiple of 8 elements, so that every layer starts 16-byte aligned);
 * attention: g,
 * Wqkv [3 H D][d], Wo [d][H D].  Layers in order, each group of attn_every
 * layers = (attn_every - 1) Mamba layers then one attention layer.
 */
typedef struct {
  int n_layers, d_model, attn_every, n_heads, head_dim, ssm_heads, ssm_head_dim, ssm_state;
  float rms_eps, rope_base;
} oracle_hybrid_cfg;

int64_t oracle_hybrid_mamba_elems(const oracle_hybrid_cfg* c) {
  const int64_t d = c->d_model, di = (int64_t)c->ssm_heads * c->ssm_head_dim;
  return d + (2 * di + 2 * c->ssm_state + c->ssm_heads) * d + d * di + (3 * (int64_t)c->ssm_heads + 7) / 8 * 8;
}
int64_t oracle_hybrid_attn_elems(const oracle_hybrid_cfg* c) {
  const int64_t d = c->d_model, HD = (int64_t)c->n_heads * c->head_dim;
  return d + 3 * HD * d + d * HD;
}
int64_t oracle_hybrid_layer_offset(const oracle_hybrid_cfg* c, int l) {
  const int64_t M = oracle_hybrid_mamba_elems(c), A = oracle_hybrid_attn_elems(c);
  const int e = c->attn_every;
  return (int64_t)(l / e) * ((e - 1) * M + A) + (int64_t)(l % e) * M;
}

static double oracle_softplus(double v) { return v > 0 ? v + log1p(exp(-v)) : log1p(exp(v)); }

/* The state update and gated output of one Mamba2-style block for one
 * session, from its in-projection output zx = [z d_i | x d_i | B N | C N |
 * dt Hs]: per head dt = softplus(dt + dt_bias), a = exp(dt * -exp(A_log)); per
 * head dim p and state n the state becomes a h + dt B[n] x[p], stored in fp32
 * (the state is fp32), y[p] = sum_n C[n] h[p][n] + D x[p] over the stored
 * values, out[p] = y[p] silu(z[p]) (unrounded).  state is [Hs][P][N]. */
void oracle_ssm_update(const oracle_hybrid_cfg* c, const double* zx, const uint16_t* a_log,
                       const uint16_t* dt_bias, const uint16_t* dskip, float* state, double* out) {
  const int Hs = c->ssm_heads, P = c->ssm_head_dim, N = c->ssm_state;
  const int di = Hs * P;
  const double* z = zx;
  const double* xs = zx + di;
  const double* B = zx + 2 * di;
  const double* C = zx + 2 * di + N;
  const double* dtr = zx + 2 * di + 2 * N;
  for (int hh = 0; hh < Hs; ++hh) {
    const double dt = oracle_softplus(dtr[hh] + oracle_bf16_to_double(dt_bias[hh]));
    const double A = -exp(oracle_bf16_to_double(a_log[hh]));
    const double a = exp(dt * A);
    const double Dh = oracle_bf16_to_double(dskip[hh]);
    for (int p = 0; p < P; ++p) {
      const double xp = xs[hh * P + p];
      float* hrow = state + ((int64_t)hh * P + p) * N;
      double acc = 0.0;
      for (int n = 0; n < N; ++n) {
        const float hn = (float)(a * (double)hrow[n] + dt * B[n] * xp);
        hrow[n] = hn;
        acc += C[n] * (double)hn;
      }
      const double y = acc + Dh * xp;
      out[hh * P + p] = y * oracle_silu(z[hh * P + p]);
    }
  }
}

/* One Mamba2-style block's mixer for one session: xn (bf16-rounded) in,
 * zx = W_in xn, then the state update and gated output above. */
void oracle_ssm_mixer(const oracle_hybrid_cfg* c, const uint16_t* w_in, const uint16_t* a_log,
                      const uint16_t* dt_bias, const uint16_t* dskip, const double* xn,
                      float* state, double* out) {
  const int d = c->d_model, di = c->ssm_heads * c->ssm_head_dim;
  const int rows = 2 * di + 2 * c->ssm_state + c->ssm_heads;
  double* zx = (double*)malloc(sizeof(double) * rows);
  oracle_matvec(w_in, rows, d, xn, zx);
  oracle_ssm_update(c, zx, a_log, dt_bias, dskip, state, out);
  free(zx);
}

/*
 * One frame of the hybrid model for n sessions.  kv / kv_scales hold the
 * attention layers' histories ([La][2][n][H][T_max][D], La = n_layers /
 * attn_every), state the Mamba layers' ([Lm][n][Hs][P][N] fp32, Lm = n_layers
 * - La), both updated in place.  Positions as in oracle_step (negative: an
 * empty slot, y = x, nothing touched).  Returns 0 or -(s+1).
 */
int oracle_hybrid_step(const oracle_hybrid_cfg* c, int T_max, const uint16_t* weights, int n, uint8_t* kv,
                       float* kv_scales, float* state, const int32_t* pos, const uint16_t* x, uint16_t* y,
                       double* y_exact) {
  const int L = c->n_layers, d = c->d_model, H = c->n_heads, D = c->head_dim, e = c->attn_every;
  const int HD = H * D, Hs = c->ssm_heads, P = c->ssm_head_dim, N = c->ssm_state, di = Hs * P;
  const int rows_in = 2 * di + 2 * N + Hs;
  for (int s = 0; s < n; ++s)
    if (pos[s] >= T_max) return -(s + 1);
  double* r = (double*)malloc(sizeof(double) * d);
  double* xn = (double*)malloc(sizeof(double) * d);
  double* qkv = (double*)malloc(sizeof(double) * 3 * HD);
  double* att = (double*)malloc(sizeof(double) * (HD > di ? HD : di));
  double* tmp = (double*)malloc(sizeof(double) * d);
  float* row = (float*)malloc(sizeof(float) * D);
  for (int s = 0; s < n; ++s) {
    const int Pp = pos[s];
    if (Pp < 0) {
      for (int i = 0; i < d; ++i) {
        y[(int64_t)s * d + i] = x[(int64_t)s * d + i];
        if (y_exact) y_exact[(int64_t)s * d + i] = oracle_bf16_to_double(x[(int64_t)s * d + i]);
      }
      continue;
    }
    for (int i = 0; i < d; ++i) r[i] = oracle_bf16_to_double(x[(int64_t)s * d + i]);
    for (int l = 0; l < L; ++l) {
      const uint16_t* Wl = weights + oracle_hybrid_layer_offset(c, l);
      oracle_rmsnorm(r, Wl, d, c->rms_eps, xn);
      for (int i = 0; i < d; ++i) xn[i] = oracle_bf16_round(xn[i]);
      if (l % e == e - 1) {
        const int la = l / e;
        const uint16_t* wqkv = Wl + d;
        const uint16_t* wo = wqkv + (int64_t)3 * HD * d;
        oracle_matvec(wqkv, 3 * HD, d, xn, qkv);
        double* q = qkv;
        double* k = qkv + HD;
        double* v = qkv + 2 * HD;
        for (int h = 0; h < H; ++h) {
          oracle_rope(q + h * D, D, Pp, c->rope_base);
          oracle_rope(k + h * D, D, Pp, c->rope_base);
        }
        for (int which = 0; which < 2; ++which) {
          const double* src = which ? v : k;
          for (int h = 0; h < H; ++h) {
            const int64_t sh = (((int64_t)la * 2 + which) * n + s) * H + h;
            for (int i = 0; i < D; ++i) row[i] = (float)src[h * D + i];
            oracle_quantize_row(row, D, kv + (sh * T_max + Pp) * D, kv_scales + sh * T_max + Pp);
          }
        }
        for (int h = 0; h < H; ++h) {
          const int64_t shk = (((int64_t)la * 2 + 0) * n + s) * H + h;
          const int64_t shv = (((int64_t)la * 2 + 1) * n + s) * H + h;
          oracle_attention_head(q + h * D, kv + shk * T_max * D, kv_scales + shk * T_max,
                                kv + shv * T_max * D, kv_scales + shv * T_max, Pp, D, att + h * D);
        }
        for (int i = 0; i < HD; ++i) att[i] = oracle_bf16_round(att[i]);
        oracle_matvec(wo, d, HD, att, tmp);
      } else {
        const int lm = l - l / e;
        const uint16_t* w_in = Wl + d;
        const uint16_t* w_out = w_in + (int64_t)rows_in * d;
        const uint16_t* a_log = w_out + (int64_t)d * di;
        float* st = state + ((int64_t)lm * n + s) * (int64_t)Hs * P * N;
        oracle_ssm_mixer(c, w_in, a_log, a_log + Hs, a_log + 2 * Hs, xn, st, att);
        for (int i = 0; i < di; ++i) att[i] = oracle_bf16_round(att[i]);
        oracle_matvec(w_out, d, di, att, tmp);
      }
      for (int i = 0; i < d; ++i) r[i] += tmp[i];
    }
    for (int i = 0; i < d; ++i) {
      y[(int64_t)s * d + i] = oracle_double_to_bf16(r[i]);
      if (y_exact) y_exact[(int64_t)s * d + i] = r[i];
    }
  }
  free(r); free(xn); free(qkv); free(att); free(tmp); free(row);
  return 0;
}
