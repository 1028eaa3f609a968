/*
 * dflash_oracle.c -- plain, slow CPU oracle for one DFlash draft-and-verify cycle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the test suite, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or constant with the CUDA
 * library: every formula below is written out again from the method's
 * description.
 *
 * Sources (web pages on DFlash; cited by page title and section):
 *  [G]  "DFlash: block-diffusion accelerated LLM speculative decoding" guide
 *       (txtmix.com), section 3.1 "one forward pass yields the whole block",
 *       section 3.2 "draft conditioned on target features", section 3.3
 *       "verification is still done by the target", section 4 "how one task
 *       flows through the system", section 7 "DFlash 2" (path selector),
 *       FAQ Q2 (where the context features come from).
 *  [N]  "DFlash 2 release: parallel drafts keep lowering LLM inference
 *       latency" (openai-hub.com news), sections "the core of DFlash 2: write
 *       one block at a time" (prefix-acceptance example) and "KV injection".
 *  [T]  "DFlash: diffusion draft models push speculative decoding ..."
 *       (llmapis.com), "data and technical details" (draft sliding window).
 *
 * Arithmetic model.  Accumulation and activations are held in double.  In
 * bf16 mode every value is rounded to bfloat16 (round-to-nearest-even, via
 * float) at the tensor boundaries where the GPU path stores bf16: the inputs
 * of every projection (post-RMSNorm activations, attention output, SiLU*up
 * product, fused context feature c_t, tap features), the query, and the K/V
 * cache entries.  The residual stream, softmax and logits are not rounded,
 * except that the argmax is taken over logits rounded to float, the
 * precision in which the GPU takes that decision.  In fp32 mode nothing is
 * rounded.  Weights are read as bf16 (uint16 bit patterns) or float.
 *
 * Compile with -ffp-contract=off so that x86 and Arm builds agree.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_CAUSAL 0
#define OR_BIDIR 1

typedef struct {
  int H;        /* hidden size */
  int nq;       /* query heads */
  int nkv;      /* key/value heads (GQA groups) */
  int d;        /* head dim */
  int I;        /* SwiGLU intermediate size */
  int bf16;     /* 1: bf16 weights + bf16 rounding points; 0: fp32 weights, no rounding */
  double theta; /* RoPE base */
  double eps;   /* RMSNorm epsilon */
} or_cfg;

/* DFlash 2 two-tap dynamic depthwise convolutions of one draft layer, at
 * OR_CONV_PRE_ATTN (the attention input), OR_CONV_POST_ATTN (the attention
 * block's output), OR_CONV_PRE_MLP, OR_CONV_POST_MLP.  w1[i] [r][H] and
 * w2[i] [2H][r] generate the taps (see or_dyn_conv). */
#define OR_CONV_PRE_ATTN 0
#define OR_CONV_POST_ATTN 1
#define OR_CONV_PRE_MLP 2
#define OR_CONV_POST_MLP 3
typedef struct {
  const void* w1[4];
  const void* w2[4];
  int r;
} or_conv;

typedef struct {
  const void *wq, *wk, *wv, *wo; /* [out][in] row-major */
  const void *wg, *wu, *wd;      /* gate [I][H], up [I][H], down [H][I] */
  const void *g1, *g2;           /* RMSNorm gains [H] before attention / before MLP */
} or_layer;

/* ---------------------------------------------------------------- scalars */

/* float -> bfloat16 -> float, round to nearest even; NaN stays NaN. */
double or_bf16_round(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) {
    u |= 0x00400000u; /* quiet NaN */
  } else {
    u += 0x7fffu + ((u >> 16) & 1u);
  }
  u &= 0xffff0000u;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double rnd(const or_cfg* c, double x) { return c->bf16 ? or_bf16_round(x) : x; }

/* Element i of a weight tensor stored as bf16 bits or float. */
static double wget(const or_cfg* c, const void* w, size_t i) {
  if (c->bf16) {
    uint32_t u = (uint32_t)((const uint16_t*)w)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  return (double)((const float*)w)[i];
}

/* ------------------------------------------------------------- primitives */

/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g  ([G] 3.2 names RMSNorm for the
 * fused feature; the decoder layers use the same pre-norm). */
void or_rmsnorm(const or_cfg* c, int n, const double* x, const void* g, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + c->eps);
  for (int i = 0; i < n; ++i) y[i] = x[i] * inv * wget(c, g, (size_t)i);
}

/* Rotary position embedding, rotate-half pairing (i, i + d/2), angle
 * pos * theta^(-2i/d), applied to one head vector in place. */
void or_rope(double* v, int d, long pos, double theta) {
  int half = d / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
    double ang = (double)pos * inv_freq;
    double cs = cos(ang), sn = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * cs - b * sn;
    v[i + half] = b * cs + a * sn;
  }
}

/* Y[m][n] = sum_k W[n][k] * X[m][k], serial k order (same arithmetic for a
 * row whatever M is). */
void or_linear(const or_cfg* c, const void* W, int N, int K, int M, const double* X,
               double* Y) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    for (int m = 0; m < M; ++m) {
      double s = 0.0;
      for (int k = 0; k < K; ++k) s += wget(c, W, (size_t)n * K + k) * X[(size_t)m * K + k];
      Y[(size_t)m * N + n] = s;
    }
  }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * DFlash 2 two-tap dynamic depthwise convolution ([G] section 7: a two-tap
 * convolution that looks at the current and the previous position only,
 * inserted before and after attention and the MLP of every draft layer; the
 * block head reads the last verified token).  The page gives neither the tap
 * generator nor the residual form; as read here, over the M rows u[0..M-1]
 * of one block at consecutive positions:
 *   z_t       = SiLU(W1 u_t)                 W1 [r][H]
 *   (a_t,b_t) = W2 z_t                       W2 [2H][r]: rows 0..H-1 -> a, H..2H-1 -> b
 *   y_t       = u_t + a_t * u_t + b_t * u_{t-1}   per channel
 * with u_{-1} = 0: block row 0 (the anchor) has no predecessor inside the
 * block, and row 1, the first drafted position, reads the anchor, which is
 * the last verified token.  The taps come from the row itself (dynamic), one
 * pair per channel (depthwise).  Nothing is rounded here.
 */
void or_dyn_conv(const or_cfg* c, int M, int r, const void* W1, const void* W2, const double* u,
                 double* y) {
  const int H = c->H;
  double* z = malloc(sizeof(double) * (size_t)r);
  for (int t = 0; t < M; ++t) {
    const double* ut = u + (size_t)t * H;
    const double* up = t > 0 ? u + (size_t)(t - 1) * H : NULL;
    for (int j = 0; j < r; ++j) {
      double s = 0.0;
      for (int k = 0; k < H; ++k) s += wget(c, W1, (size_t)j * H + k) * ut[k];
      z[j] = silu(s);
    }
    for (int ch = 0; ch < H; ++ch) {
      double a = 0.0, b = 0.0;
      for (int j = 0; j < r; ++j) {
        a += wget(c, W2, (size_t)ch * r + j) * z[j];
        b += wget(c, W2, (size_t)(H + ch) * r + j) * z[j];
      }
      y[(size_t)t * H + ch] = ut[ch] + a * ut[ch] + (up ? b * up[ch] : 0.0);
    }
  }
  free(z);
}

/* rows u[M][H] -> conv (in place through a scratch copy) */
static void conv_rows(const or_cfg* c, const or_conv* cv, int at, int M, double* u, int round_out) {
  const int H = c->H;
  double* y = malloc(sizeof(double) * (size_t)M * H);
  or_dyn_conv(c, M, cv->r, cv->w1[at], cv->w2[at], u, y);
  for (size_t i = 0; i < (size_t)M * H; ++i) u[i] = round_out ? rnd(c, y[i]) : y[i];
  free(y);
}

/* Softmax attention of one query head over nk keys (pointers to head rows). */
static void attend(int d, const double* q, int nk, const double* const* K, const double* const* V,
                   double* out, double* scratch) {
  double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int j = 0; j < nk; ++j) {
    double s = 0.0;
    for (int e = 0; e < d; ++e) s += q[e] * K[j][e];
    s *= scale;
    scratch[j] = s;
    if (s > mx) mx = s;
  }
  double den = 0.0;
  for (int j = 0; j < nk; ++j) {
    scratch[j] = exp(scratch[j] - mx);
    den += scratch[j];
  }
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  for (int j = 0; j < nk; ++j) {
    double p = scratch[j] / den;
    for (int e = 0; e < d; ++e) out[e] += p * V[j][e];
  }
}

/* Slot of absolute position t in a context cache: plain index, or a ring of
 * `window` slots when the draft sliding window is on ([T]). */
static long slot_of(long t, long window) { return window > 0 ? t % window : t; }

/* --------------------------------------------------------- decoder layer */

/*
 * One pre-norm decoder layer (RMSNorm -> QKV -> RoPE -> GQA attention -> O +
 * residual -> RMSNorm -> SwiGLU MLP + residual) over M rows of ONE sequence
 * at consecutive positions p0 .. p0+M-1.  h [M][H] is the residual stream,
 * updated in place.  Caches are [nkv][cap][d].
 *
 * mode OR_CAUSAL (target verification, [G] 3.3): the rows' K/V are written
 * into the cache at their positions first, and row i attends cache positions
 * 0 .. p0+i.
 *
 * mode OR_BIDIR (draft block, [G] 3.1/3.2): the cache holds the injected
 * context K/V of positions lo .. p0-1 (lo = max(0, p0-window) with a window,
 * else 0); row i attends all of those and all M rows of the block, with no
 * mask inside the block.  The block K/V are not stored.
 */
/*
 * Stage values of one layer, each [M][width] row-major: x1 = the attention
 * input (rounded RMSNorm), q = rotated queries, k / v = the rows' rotated
 * keys and values ([M][nkv*d]), o = the attention output, x2 = the MLP input,
 * act = SiLU(gate)*up.  Any field may be NULL.
 */
typedef struct {
  double *x1, *q, *k, *v, *o, *x2, *act;
} or_stages;

static void stage_io(const double* given, double* out, double* cur, size_t n) {
  if (out) memcpy(out, cur, sizeof(double) * n);
  if (given) memcpy(cur, given, sizeof(double) * n);
}

/*
 * The layer with every stage open to inspection (teacher forcing).  When
 * out->F is non-NULL it receives this layer's own value of stage F, computed
 * from the stages before it; when given->F is non-NULL, that value then
 * replaces stage F for everything after it -- so each stage can be checked
 * against an implementation fed that implementation's own inputs.  With both
 * NULL this is exactly the plain layer.  In causal mode the cache receives
 * the (possibly given) k, v.
 */
int or_decoder_layer_tf(const or_cfg* c, const or_layer* L, const or_conv* cv, int M, long p0, int mode,
                        double* kc, double* vc, long cap, long window, double* h, const or_stages* given,
                        or_stages* out);

int or_decoder_layer_conv(const or_cfg* c, const or_layer* L, const or_conv* cv, int M, long p0,
                          int mode, double* kc, double* vc, long cap, long window, double* h) {
  return or_decoder_layer_tf(c, L, cv, M, p0, mode, kc, vc, cap, window, h, NULL, NULL);
}

int or_decoder_layer_tf(const or_cfg* c, const or_layer* L, const or_conv* cv, int M, long p0, int mode,
                        double* kc, double* vc, long cap, long window, double* h, const or_stages* given,
                        or_stages* out) {
  const or_stages none = {0, 0, 0, 0, 0, 0, 0};
  if (!given) given = &none;
  or_stages discard = none;
  if (!out) out = &discard;
  const int H = c->H, d = c->d, nq = c->nq, nkv = c->nkv, I = c->I;
  const int QD = nq * d, KD = nkv * d, grp = nq / nkv;
  if (M <= 0) return 0;
  if (mode == OR_CAUSAL && p0 + M > cap) return -1;
  if (mode == OR_BIDIR && window <= 0 && p0 > cap) return -1;
  if (mode == OR_BIDIR && window > 0 && window > cap) return -1;

  double* x = malloc(sizeof(double) * (size_t)M * H);
  double* q = malloc(sizeof(double) * (size_t)M * QD);
  double* k = malloc(sizeof(double) * (size_t)M * KD);
  double* v = malloc(sizeof(double) * (size_t)M * KD);
  double* o = malloc(sizeof(double) * (size_t)M * QD);
  double* y = malloc(sizeof(double) * (size_t)M * (H > I ? H : I));
  double* gt = malloc(sizeof(double) * (size_t)M * I);
  double* up = malloc(sizeof(double) * (size_t)M * I);
  if (!x || !q || !k || !v || !o || !y || !gt || !up) return -2;

  for (int m = 0; m < M; ++m) {
    or_rmsnorm(c, H, h + (size_t)m * H, L->g1, x + (size_t)m * H);
    for (int i = 0; i < H; ++i) x[(size_t)m * H + i] = rnd(c, x[(size_t)m * H + i]);
  }
  if (cv) conv_rows(c, cv, OR_CONV_PRE_ATTN, M, x, 1); /* a projection input: rounded */
  stage_io(given->x1, out->x1, x, (size_t)M * H);
  or_linear(c, L->wq, QD, H, M, x, q);
  or_linear(c, L->wk, KD, H, M, x, k);
  or_linear(c, L->wv, KD, H, M, x, v);
  for (int m = 0; m < M; ++m) {
    long pos = p0 + m;
    for (int hh = 0; hh < nq; ++hh) or_rope(q + (size_t)m * QD + (size_t)hh * d, d, pos, c->theta);
    for (int hh = 0; hh < nkv; ++hh) or_rope(k + (size_t)m * KD + (size_t)hh * d, d, pos, c->theta);
    for (int i = 0; i < QD; ++i) q[(size_t)m * QD + i] = rnd(c, q[(size_t)m * QD + i]);
    for (int i = 0; i < KD; ++i) {
      k[(size_t)m * KD + i] = rnd(c, k[(size_t)m * KD + i]);
      v[(size_t)m * KD + i] = rnd(c, v[(size_t)m * KD + i]);
    }
  }
  stage_io(given->q, out->q, q, (size_t)M * QD);
  stage_io(given->k, out->k, k, (size_t)M * KD);
  stage_io(given->v, out->v, v, (size_t)M * KD);
  if (mode == OR_CAUSAL) {
    for (int m = 0; m < M; ++m)
      for (int g = 0; g < nkv; ++g) {
        memcpy(kc + ((size_t)g * cap + (size_t)(p0 + m)) * d, k + (size_t)m * KD + (size_t)g * d,
               sizeof(double) * d);
        memcpy(vc + ((size_t)g * cap + (size_t)(p0 + m)) * d, v + (size_t)m * KD + (size_t)g * d,
               sizeof(double) * d);
      }
  }

  long lo = (mode == OR_BIDIR && window > 0) ? (p0 > window ? p0 - window : 0) : 0;
  long maxk = (mode == OR_CAUSAL) ? (p0 + M) : (p0 - lo + M);
#pragma omp parallel
  {
    const double** Kp = malloc(sizeof(double*) * (size_t)maxk);
    const double** Vp = malloc(sizeof(double*) * (size_t)maxk);
    double* sc = malloc(sizeof(double) * (size_t)maxk);
#pragma omp for schedule(static)
    for (int mh = 0; mh < M * nq; ++mh) {
      int m = mh / nq, hq = mh % nq, g = hq / grp;
      int nk = 0;
      if (mode == OR_CAUSAL) {
        for (long t = 0; t <= p0 + m; ++t) {
          Kp[nk] = kc + ((size_t)g * cap + (size_t)t) * d;
          Vp[nk] = vc + ((size_t)g * cap + (size_t)t) * d;
          ++nk;
        }
      } else {
        for (long t = lo; t < p0; ++t) {
          Kp[nk] = kc + ((size_t)g * cap + (size_t)slot_of(t, window)) * d;
          Vp[nk] = vc + ((size_t)g * cap + (size_t)slot_of(t, window)) * d;
          ++nk;
        }
        for (int j = 0; j < M; ++j) {
          Kp[nk] = k + (size_t)j * KD + (size_t)g * d;
          Vp[nk] = v + (size_t)j * KD + (size_t)g * d;
          ++nk;
        }
      }
      attend(d, q + (size_t)m * QD + (size_t)hq * d, nk, Kp, Vp, o + (size_t)m * QD + (size_t)hq * d,
             sc);
    }
    free(Kp);
    free(Vp);
    free(sc);
  }
  for (size_t i = 0; i < (size_t)M * QD; ++i) o[i] = rnd(c, o[i]);
  stage_io(given->o, out->o, o, (size_t)M * QD);

  or_linear(c, L->wo, H, QD, M, o, y);
  if (cv) conv_rows(c, cv, OR_CONV_POST_ATTN, M, y, 0); /* added to the residual: not rounded */
  for (size_t i = 0; i < (size_t)M * H; ++i) h[i] += y[i];

  for (int m = 0; m < M; ++m) {
    or_rmsnorm(c, H, h + (size_t)m * H, L->g2, x + (size_t)m * H);
    for (int i = 0; i < H; ++i) x[(size_t)m * H + i] = rnd(c, x[(size_t)m * H + i]);
  }
  if (cv) conv_rows(c, cv, OR_CONV_PRE_MLP, M, x, 1);
  stage_io(given->x2, out->x2, x, (size_t)M * H);
  or_linear(c, L->wg, I, H, M, x, gt);
  or_linear(c, L->wu, I, H, M, x, up);
  for (size_t i = 0; i < (size_t)M * I; ++i) gt[i] = rnd(c, silu(gt[i]) * up[i]);
  stage_io(given->act, out->act, gt, (size_t)M * I);
  or_linear(c, L->wd, H, I, M, gt, y);
  if (cv) conv_rows(c, cv, OR_CONV_POST_MLP, M, y, 0);
  for (size_t i = 0; i < (size_t)M * H; ++i) h[i] += y[i];

  free(x); free(q); free(k); free(v); free(o); free(y); free(gt); free(up);
  return 0;
}

/* The layer without the DFlash 2 convolutions. */
int or_decoder_layer(const or_cfg* c, const or_layer* L, int M, long p0, int mode,
                     double* kc, double* vc, long cap, long window, double* h) {
  return or_decoder_layer_conv(c, L, NULL, M, p0, mode, kc, vc, cap, window, h);
}

/* ------------------------------------------------------------ output head */

/* x_out[m] = round(RMSNorm(h[m]; g)) -- the final norm before the LM head. */
void or_final_norm(const or_cfg* c, int M, const double* h, const void* g, double* x_out) {
  for (int m = 0; m < M; ++m) {
    or_rmsnorm(c, c->H, h + (size_t)m * c->H, g, x_out + (size_t)m * c->H);
    for (int i = 0; i < c->H; ++i) x_out[(size_t)m * c->H + i] = rnd(c, x_out[(size_t)m * c->H + i]);
  }
}

/*
 * LM head + greedy argmax: logit[m][v] = W_lm[v] . x[m]; argmax over the
 * float-rounded logits, lowest vocab index on ties; margin = top1 - top2
 * (0 for an exact tie).  logits (optional, [M][V]) receives the float logits.
 */
void or_lm_head_argmax(const or_cfg* c, const void* Wlm, int V, int M, const double* x,
                       int* argmax, double* margin, float* logits) {
  const int H = c->H;
  for (int m = 0; m < M; ++m) {
    float* row = malloc(sizeof(float) * (size_t)V);
#pragma omp parallel for schedule(static)
    for (int t = 0; t < V; ++t) {
      double s = 0.0;
      for (int k = 0; k < H; ++k) s += wget(c, Wlm, (size_t)t * H + k) * x[(size_t)m * H + k];
      row[t] = (float)s;
    }
    int best = 0;
    for (int t = 1; t < V; ++t)
      if (row[t] > row[best]) best = t;
    double second = -INFINITY;
    for (int t = 0; t < V; ++t)
      if (t != best && (double)row[t] > second) second = (double)row[t];
    argmax[m] = best;
    margin[m] = (double)row[best] - second;
    if (logits) memcpy(logits + (size_t)m * V, row, sizeof(float) * (size_t)V);
    free(row);
  }
}

/* -------------------------------------------------------------- acceptance */

/*
 * Greedy longest-prefix acceptance ([N] prefix example: 8 drafted, 6 agree,
 * decoding resumes at the 7th from the target; [G] section 4 step 4).
 * drafts[j-1] is the draft for block row j (j = 1..B-1); g[i] is the target's
 * greedy token after block row i (i = 0..B-1).  Draft j is accepted while it
 * equals g[j-1]; the bonus token is g[k] after k accepted drafts.
 * out_tokens[0..k-1] = accepted drafts, out_tokens[k] = bonus.  Returns k.
 */
int or_accept(int B, const int* drafts, const int* g, int* out_tokens) {
  int k = 0;
  while (k < B - 1 && drafts[k] == g[k]) {
    out_tokens[k] = drafts[k];
    ++k;
  }
  out_tokens[k] = g[k];
  return k;
}

/* ---------------------------------------------- context fusion + injection */

/*
 * Context-feature fusion and KV injection ([G] 3.2 and FAQ Q2; [N] "KV
 * injection"): for each position t with tap features f_t = [h_t^{l_1}, ...,
 * h_t^{l_F}] (already rounded, [T][F*H]),
 *     c_t = round(RMSNorm(W_fc f_t; g_fc)),
 * and for every draft layer j
 *     K_ctx^j[t] = round(RoPE(W_k^j c_t, t)),  V_ctx^j[t] = round(W_v^j c_t),
 * written to slot slot_of(t, window) of the layer's context cache [nkv][cap][d].
 * c_out (optional, [T][H]) receives c_t.
 */
int or_fuse_context(const or_cfg* c, int F, const void* Wfc, const void* gfc, int T,
                    const double* feats, const long* pos, int n_layers, const void* const* wk,
                    const void* const* wv, double* const* kc, double* const* vc, long cap,
                    long window, double* c_out) {
  const int H = c->H, d = c->d, nkv = c->nkv, KD = nkv * d;
  double* z = malloc(sizeof(double) * (size_t)T * H);
  double* cc = malloc(sizeof(double) * (size_t)T * H);
  double* kk = malloc(sizeof(double) * (size_t)T * KD);
  double* vv = malloc(sizeof(double) * (size_t)T * KD);
  if (!z || !cc || !kk || !vv) return -2;
  for (int t = 0; t < T; ++t) {
    long s = slot_of(pos[t], window);
    if (pos[t] < 0 || s >= cap) return -1;
  }
  or_linear(c, Wfc, H, F * H, T, feats, z);
  for (int t = 0; t < T; ++t) {
    or_rmsnorm(c, H, z + (size_t)t * H, gfc, cc + (size_t)t * H);
    for (int i = 0; i < H; ++i) cc[(size_t)t * H + i] = rnd(c, cc[(size_t)t * H + i]);
  }
  if (c_out) memcpy(c_out, cc, sizeof(double) * (size_t)T * H);
  for (int j = 0; j < n_layers; ++j) {
    or_linear(c, wk[j], KD, H, T, cc, kk);
    or_linear(c, wv[j], KD, H, T, cc, vv);
    for (int t = 0; t < T; ++t) {
      long s = slot_of(pos[t], window);
      for (int g = 0; g < nkv; ++g) {
        double* kr = kk + (size_t)t * KD + (size_t)g * d;
        or_rope(kr, d, pos[t], c->theta);
        for (int e = 0; e < d; ++e) {
          kc[j][((size_t)g * cap + (size_t)s) * d + e] = rnd(c, kr[e]);
          vc[j][((size_t)g * cap + (size_t)s) * d + e] = rnd(c, vv[(size_t)t * KD + (size_t)g * d + e]);
        }
      }
    }
  }
  free(z); free(cc); free(kk); free(vv);
  return 0;
}

/* ----------------------------------------------------------- path selector */

/*
 * DFlash 2 path selector ([G] section 7), greedy form.  For each block row
 * j = 1..B-1 keep the top-`topk` draft candidates of that row's logits
 * (ordered by logit descending, index ascending).  The score of a transition
 * a -> b is the low-rank bilinear form (U e_a) . (V e_b) with e the shared
 * embedding rows and U, Vm in R^{R x H}.  Walk greedily: p_0 = anchor,
 * p_j = the candidate of row j with the highest score from p_{j-1}, the
 * lower rank on ties.  logits: [B-1][Vocab] float (row j-1 for block row j).
 * path[j-1] = p_j; cand [B-1][topk] receives the candidate lists; margin[j-1]
 * = best minus second-best score at step j.
 */
void or_path_select(const or_cfg* c, int B, int Vocab, int topk, int R, const float* logits,
                    const void* E, const void* U, const void* Vm, int anchor, int* cand,
                    int* path, double* margin) {
  const int H = c->H;
  double* ue = malloc(sizeof(double) * (size_t)R);
  double* ve = malloc(sizeof(double) * (size_t)R);
  for (int j = 0; j < B - 1; ++j) {
    const float* row = logits + (size_t)j * Vocab;
    int* cj = cand + (size_t)j * topk;
    for (int r = 0; r < topk; ++r) {
      int best = -1;
      for (int t = 0; t < Vocab; ++t) {
        int used = 0;
        for (int q = 0; q < r; ++q)
          if (cj[q] == t) used = 1;
        if (used) continue;
        if (best < 0 || row[t] > row[best]) best = t;
      }
      cj[r] = best;
    }
  }
  int prev = anchor;
  for (int j = 0; j < B - 1; ++j) {
    for (int r = 0; r < R; ++r) {
      double s = 0.0;
      for (int k = 0; k < H; ++k) s += wget(c, U, (size_t)r * H + k) * wget(c, E, (size_t)prev * H + k);
      ue[r] = s;
    }
    double best = -INFINITY, second = -INFINITY;
    int bi = 0;
    for (int q = 0; q < topk; ++q) {
      int b = cand[(size_t)j * topk + q];
      double sc = 0.0;
      for (int r = 0; r < R; ++r) {
        double s = 0.0;
        for (int k = 0; k < H; ++k) s += wget(c, Vm, (size_t)r * H + k) * wget(c, E, (size_t)b * H + k);
        ve[r] = s;
        sc += ue[r] * ve[r];
      }
      sc = (double)(float)sc; /* decided in float, the precision of the GPU path */
      if (sc > best) {
        second = best;
        best = sc;
        bi = q;
      } else if (sc > second) {
        second = sc;
      }
    }
    path[j] = cand[(size_t)j * topk + bi];
    margin[j] = best - second;
    prev = path[j];
  }
  free(ue);
  free(ve);
}

/* ------------------------------------------------------------- sampling
 *
 * Sampling-mode verification, the lossless-in-distribution variant of the
 * greedy rule ([G] section 7: the path is walked "greedily or by sampling"
 * and rejection sampling keeps the output distribution exactly the
 * target's).  This follows speculative sampling as published (Leviathan,
 * Kalman, Matias, "Fast Inference from Transformers via Speculative
 * Decoding", ICML 2023; Chen et al., "Accelerating Large Language Model
 * Decoding with Speculative Sampling", 2023) at temperature T:
 *   p_j = softmax(target logits of block row j / T), q_j = softmax(draft
 *   logits of block row j+1 / T) -- both the distribution of the token at
 *   position P+j+1;
 *   the draft token d of block row j+1 is sampled from q_j;
 *   it is accepted with probability min(1, p_j(d) / q_j(d)), i.e. iff
 *   log u < log p_j(d) - log q_j(d);
 *   at the first rejection the emitted token is sampled from
 *   max(0, p_j - q_j) normalised; if every draft is accepted a bonus token
 *   is sampled from the last target row.
 * A categorical draw from weights w is the argmax over v of log w_v + g_v
 * (Gumbel-max; exponential race for unnormalised weights), g_v Gumbel(0,1).
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11), key (seed low, seed high),
 * counter (vocabulary entry, position, sequence << 8 | purpose, cycle);
 * u = ((x0 >> 8) + 1/2) 2^-24 in (0, 1), g = -log(-log u).
 */
enum { OR_RNG_DRAFT = 1, OR_RNG_ACCEPT = 2, OR_RNG_RESID = 3, OR_RNG_BONUS = 4, OR_RNG_PATH = 5 };

void or_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u; /* Weyl key schedule */
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

double or_uniform(uint64_t seed, uint32_t v, uint32_t pos, uint32_t seq, uint32_t purpose, uint32_t cycle) {
  const uint32_t ctr[4] = {v, pos, (seq << 8) | (purpose & 0xFFu), cycle};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t x[4];
  or_philox4x32_10(ctr, key, x);
  return ((double)(x[0] >> 8) + 0.5) * (1.0 / 16777216.0);
}

static double gumbel(uint64_t seed, uint32_t v, uint32_t pos, uint32_t seq, uint32_t purpose, uint32_t cycle) {
  return -log(-log(or_uniform(seed, v, pos, seq, purpose, cycle)));
}

/* ------------------------------------------------- top-k / top-p filter
 *
 * The pages name sampling but no filter; the usual one is read here.  The
 * entries of a row are ordered by logit (descending; lower index first on
 * equal logits), which is the order of l / T for any T > 0.  top_k > 0
 * keeps the first top_k; then top_p < 1 keeps the shortest prefix of those
 * whose probability mass, softmax(l / T) renormalised over them, reaches
 * top_p.  keep[v] = 1 for the kept entries; returns their number.  *pmargin
 * (near-tie reporting) = the smallest |cumulative mass - top_p| on either
 * side of the top-p boundary, +inf when top-p is off.
 */
static const float* g_sort_row;
static int by_logit_desc(const void* x, const void* y) {
  const int a = *(const int*)x, b = *(const int*)y;
  const float la = g_sort_row[a], lb = g_sort_row[b];
  if (la > lb) return -1;
  if (la < lb) return 1;
  return a < b ? -1 : (a > b ? 1 : 0);
}

int or_filter_row(const float* l, int V, double T, int top_k, double top_p, unsigned char* keep,
                  double* pmargin) {
  if (V <= 0) return 0;
  int* order = malloc(sizeof(int) * (size_t)V);
  for (int v = 0; v < V; ++v) order[v] = v;
  g_sort_row = l;
  qsort(order, (size_t)V, sizeof(int), by_logit_desc);
  int n = (top_k > 0 && top_k < V) ? top_k : V;
  double mg = INFINITY;
  if (top_p < 1.0) {
    const double mx = (double)l[order[0]] / T;
    double z = 0.0;
    for (int i = 0; i < n; ++i) z += exp((double)l[order[i]] / T - mx);
    double cum = 0.0;
    int cut = n;
    for (int i = 0; i < n; ++i) {
      const double before = cum;
      cum += exp((double)l[order[i]] / T - mx);
      if (cum >= top_p * z) {
        cut = i + 1;
        mg = fmin(fabs(before / z - top_p), fabs(cum / z - top_p));
        break;
      }
    }
    n = cut;
  }
  memset(keep, 0, (size_t)V);
  for (int i = 0; i < n; ++i) keep[order[i]] = 1;
  free(order);
  if (pmargin) *pmargin = mg;
  return n;
}

/* log sum_v exp(l_v / T) over the kept entries (keep == NULL: all) */
static double row_lse_k(const float* l, int V, double T, const unsigned char* keep) {
  double mx = -INFINITY;
  for (int v = 0; v < V; ++v)
    if (!keep || keep[v]) mx = fmax(mx, (double)l[v] / T);
  double s = 0.0;
  for (int v = 0; v < V; ++v)
    if (!keep || keep[v]) s += exp((double)l[v] / T - mx);
  return mx + log(s);
}

/* A draw from softmax(l / T) restricted to the kept entries (keep == NULL:
 * all): argmax_v l_v / T + g_v (lowest index on ties).  Returns the token;
 * *lse = log sum exp(l / T) over the kept entries; *margin = best - second. */
int or_sample_row_f(const float* l, int V, double T, const unsigned char* keep, uint64_t seed, int pos, int seq,
                    int purpose, int cycle, double* lse, double* margin) {
  int bi = -1;
  double best = -INFINITY, second = -INFINITY;
  for (int v = 0; v < V; ++v) {
    if (keep && !keep[v]) continue;
    const double sc = (double)l[v] / T + gumbel(seed, (uint32_t)v, (uint32_t)pos, (uint32_t)seq, (uint32_t)purpose,
                                                (uint32_t)cycle);
    if (bi < 0 || sc > best) {
      second = best;
      best = sc;
      bi = v;
    } else if (sc > second) {
      second = sc;
    }
  }
  if (lse) *lse = row_lse_k(l, V, T, keep);
  if (margin) *margin = best - second;
  return bi;
}

int or_sample_row(const float* l, int V, double T, uint64_t seed, int pos, int seq, int purpose, int cycle,
                  double* lse, double* margin) {
  return or_sample_row_f(l, V, T, NULL, seed, pos, seq, purpose, cycle, lse, margin);
}

/* One sequence's block: target logits tl [B][V] (row j: position P+j+1),
 * draft logits dl [B-1][V] (row i: block row i+1, position P+i+1), drafts
 * [B-1]; keep_t [B][V] / keep_d [B-1][V] the filtered entries of each row
 * (NULL: all).  p and q are the filtered, renormalised softmax(l / T): an
 * entry outside its row's kept set has probability 0.  Writes
 * out_tokens[0..k] and returns the accept length k.  *margin = the smallest
 * decision margin met (acceptance tests and the final draw), for near-tie
 * reporting. */
int or_spec_sample_accept_f(int B, int V, const float* tl, const float* dl, const unsigned char* keep_t,
                            const unsigned char* keep_d, const int* drafts, double T, uint64_t seed, int seq, int P,
                            int cycle, int* out_tokens, double* margin) {
  double mg = INFINITY;
  int k = 0;
  for (int j = 1; j <= B - 1; ++j) {
    const int d = drafts[j - 1];
    const float* trow = tl + (size_t)(j - 1) * V;
    const float* drow = dl + (size_t)(j - 1) * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)(j - 1) * V : NULL;
    const unsigned char* kd = keep_d ? keep_d + (size_t)(j - 1) * V : NULL;
    const double lp = (kt && !kt[d]) ? -INFINITY : (double)trow[d] / T - row_lse_k(trow, V, T, kt);
    const double lq = (double)drow[d] / T - row_lse_k(drow, V, T, kd);
    const double lu = log(or_uniform(seed, 0u, (uint32_t)(P + j), (uint32_t)seq, OR_RNG_ACCEPT, (uint32_t)cycle));
    if (lp > -INFINITY) mg = fmin(mg, fabs(lu - (lp - lq)));
    if (!(lu < lp - lq)) break;
    out_tokens[k++] = d;
  }
  int x = -1;
  double best = -INFINITY, second = -INFINITY;
  if (k < B - 1) {
    /* residual max(0, p - q) at the rejected row, by exponential race */
    const float* trow = tl + (size_t)k * V;
    const float* drow = dl + (size_t)k * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)k * V : NULL;
    const unsigned char* kd = keep_d ? keep_d + (size_t)k * V : NULL;
    const double lt = row_lse_k(trow, V, T, kt), ld = row_lse_k(drow, V, T, kd);
    for (int v = 0; v < V; ++v) {
      if (kt && !kt[v]) continue; /* p = 0: weight 0 */
      const double a = (double)trow[v] / T - lt;
      const double b = (kd && !kd[v]) ? -INFINITY : (double)drow[v] / T - ld;
      if (!(a > b)) continue; /* weight 0 */
      const double sc = (b == -INFINITY ? a : a + log1p(-exp(b - a))) +
                        gumbel(seed, (uint32_t)v, (uint32_t)(P + k + 1), (uint32_t)seq, OR_RNG_RESID, (uint32_t)cycle);
      if (x < 0 || sc > best) {
        second = best;
        best = sc;
        x = v;
      } else if (sc > second) {
        second = sc;
      }
    }
  }
  if (x < 0) {
    /* all drafts accepted (or p <= q everywhere at the rejected row): a draw from p */
    const int row = k < B - 1 ? k : B - 1;
    const int purpose = k < B - 1 ? OR_RNG_RESID : OR_RNG_BONUS;
    const float* trow = tl + (size_t)row * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)row * V : NULL;
    for (int v = 0; v < V; ++v) {
      if (kt && !kt[v]) continue;
      const double sc = (double)trow[v] / T +
                        gumbel(seed, (uint32_t)v, (uint32_t)(P + row + 1), (uint32_t)seq, (uint32_t)purpose, (uint32_t)cycle);
      if (x < 0 || sc > best) {
        second = best;
        best = sc;
        x = v;
      } else if (sc > second) {
        second = sc;
      }
    }
  }
  out_tokens[k] = x;
  mg = fmin(mg, best - second);
  if (margin) *margin = mg;
  return k;
}

int or_spec_sample_accept(int B, int V, const float* tl, const float* dl, const int* drafts, double T,
                          uint64_t seed, int seq, int P, int cycle, int* out_tokens, double* margin) {
  return or_spec_sample_accept_f(B, V, tl, dl, NULL, NULL, drafts, T, seed, seq, P, cycle, out_tokens, margin);
}

/* ------------------------------------------------- sampled path walk
 *
 * The DFlash 2 path walked by sampling ([G] section 7: the path is walked
 * "greedily or by sampling" along the pair scores, and rejection sampling
 * keeps the output distribution exactly the target's).  Read here: at step
 * j (block row j+1) the proposal over row j's candidates is
 *   q_j(c) = softmax over the topk candidates c of s(p_{j-1}, c) / T,
 * s(a, b) = (U e_a) . (V e_b) the low-rank pair score of the greedy walk,
 * p_0 = anchor; p_j is a Gumbel-max draw from q_j (Philox purpose
 * OR_RNG_PATH, counter entry = the candidate's rank, position P + j + 1),
 * lower rank on equal draw scores.  The tokens outside the candidates have
 * proposal probability 0.  cand [B-1][topk] in; path [B-1], logq
 * [B-1][topk] (log q_j per candidate) and margin [B-1] (best - second draw
 * score) out.
 */
static double pair_score(const or_cfg* c, int R, const void* E, const void* U, const void* Vm, int a, int b) {
  const int H = c->H;
  double sc = 0.0;
  for (int r = 0; r < R; ++r) {
    double ua = 0.0, vb = 0.0;
    for (int k = 0; k < H; ++k) {
      ua += wget(c, U, (size_t)r * H + k) * wget(c, E, (size_t)a * H + k);
      vb += wget(c, Vm, (size_t)r * H + k) * wget(c, E, (size_t)b * H + k);
    }
    sc += ua * vb;
  }
  return sc;
}

void or_path_walk_sample(const or_cfg* c, int B, int topk, int R, const int* cand, const void* E, const void* U,
                         const void* Vm, int anchor, double T, uint64_t seed, int seq, int P, int cycle, int* path,
                         double* logq, double* margin) {
  double* z = malloc(sizeof(double) * (size_t)topk);
  int prev = anchor;
  for (int j = 0; j < B - 1; ++j) {
    double mx = -INFINITY;
    for (int q = 0; q < topk; ++q) {
      z[q] = pair_score(c, R, E, U, Vm, prev, cand[(size_t)j * topk + q]) / T;
      mx = fmax(mx, z[q]);
    }
    double sum = 0.0;
    for (int q = 0; q < topk; ++q) sum += exp(z[q] - mx);
    const double lse = mx + log(sum);
    double best = -INFINITY, second = -INFINITY;
    int bi = 0;
    for (int q = 0; q < topk; ++q) {
      logq[(size_t)j * topk + q] = z[q] - lse;
      const double sc = z[q] + gumbel(seed, (uint32_t)q, (uint32_t)(P + j + 1), (uint32_t)seq, OR_RNG_PATH,
                                      (uint32_t)cycle);
      if (sc > best) {
        second = best;
        best = sc;
        bi = q;
      } else if (sc > second) {
        second = sc;
      }
    }
    path[j] = cand[(size_t)j * topk + bi];
    margin[j] = best - second;
    prev = path[j];
  }
  free(z);
}

/* Speculative sampling against a sparse proposal: q_j is supported on the
 * candidates qc [B-1][K] with log-probabilities lq [B-1][K] (the sampled
 * walk's); everything else is as or_spec_sample_accept_f, whose target
 * filtering keep_t (NULL: none) applies. */
int or_spec_sample_accept_sparse(int B, int V, const float* tl, const unsigned char* keep_t, int K, const int* qc,
                                 const double* lq, const int* drafts, double T, uint64_t seed, int seq, int P,
                                 int cycle, int* out_tokens, double* margin) {
  double mg = INFINITY;
  int k = 0;
  for (int j = 1; j <= B - 1; ++j) {
    const int d = drafts[j - 1];
    const float* trow = tl + (size_t)(j - 1) * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)(j - 1) * V : NULL;
    const double lp = (kt && !kt[d]) ? -INFINITY : (double)trow[d] / T - row_lse_k(trow, V, T, kt);
    double lqd = -INFINITY;
    for (int q = 0; q < K; ++q)
      if (qc[(size_t)(j - 1) * K + q] == d) {
        lqd = lq[(size_t)(j - 1) * K + q];
        break;
      }
    const double lu = log(or_uniform(seed, 0u, (uint32_t)(P + j), (uint32_t)seq, OR_RNG_ACCEPT, (uint32_t)cycle));
    if (lp > -INFINITY && lqd > -INFINITY) mg = fmin(mg, fabs(lu - (lp - lqd)));
    if (!(lu < lp - lqd)) break;
    out_tokens[k++] = d;
  }
  int x = -1;
  double best = -INFINITY, second = -INFINITY;
  if (k < B - 1) {
    const float* trow = tl + (size_t)k * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)k * V : NULL;
    const double lt = row_lse_k(trow, V, T, kt);
    for (int v = 0; v < V; ++v) {
      if (kt && !kt[v]) continue;
      const double a = (double)trow[v] / T - lt;
      double b = -INFINITY;
      for (int q = 0; q < K; ++q)
        if (qc[(size_t)k * K + q] == v) {
          b = lq[(size_t)k * K + q];
          break;
        }
      if (!(a > b)) continue;
      const double sc = (b == -INFINITY ? a : a + log1p(-exp(b - a))) +
                        gumbel(seed, (uint32_t)v, (uint32_t)(P + k + 1), (uint32_t)seq, OR_RNG_RESID, (uint32_t)cycle);
      if (x < 0 || sc > best) {
        second = best;
        best = sc;
        x = v;
      } else if (sc > second) {
        second = sc;
      }
    }
  }
  if (x < 0) {
    const int row = k < B - 1 ? k : B - 1;
    const int purpose = k < B - 1 ? OR_RNG_RESID : OR_RNG_BONUS;
    const float* trow = tl + (size_t)row * V;
    const unsigned char* kt = keep_t ? keep_t + (size_t)row * V : NULL;
    for (int v = 0; v < V; ++v) {
      if (kt && !kt[v]) continue;
      const double sc = (double)trow[v] / T +
                        gumbel(seed, (uint32_t)v, (uint32_t)(P + row + 1), (uint32_t)seq, (uint32_t)purpose, (uint32_t)cycle);
      if (x < 0 || sc > best) {
        second = best;
        best = sc;
        x = v;
      } else if (sc > second) {
        second = sc;
      }
    }
  }
  out_tokens[k] = x;
  mg = fmin(mg, best - second);
  if (margin) *margin = mg;
  return k;
}

/* Threads the OpenMP loops use from now on (the CPU baseline is timed at one
 * thread and at all cores); the loops are parallel over independent output
 * rows with every reduction serial, so results do not depend on it. */
void or_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
