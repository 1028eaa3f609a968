// abi.cu -- the C ABI (include/dflash.h): host-side argument checks,
// workspace carving and the launch sequence of each entry point.  Every
// check runs before the first launch of a call; no exception crosses the ABI.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "trace.h"

using namespace dfl;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

#define DF_CHECK(cond, ...)                                 \
  do {                                                      \
    if (!(cond)) return fail(DFLASH_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define DF_CUDA(call)                                                                       \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) return fail(DFLASH_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

// Launch with optional tracing (family, algorithmic bytes).
#define DF_LAUNCH(st, fam, bytes, call)                                                     \
  do {                                                                                      \
    trace_pre((st), (fam));                                                                 \
    cudaError_t e_ = (call);                                                                \
    trace_post((st), (double)(bytes));                                                      \
    if (e_ != cudaSuccess) return fail(DFLASH_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

size_t elem_size(int dtype) { return dtype == DFLASH_BF16 ? 2 : 4; }

// Carves a workspace into 256-byte aligned pieces; with base == nullptr it
// only measures.
struct Bump {
  char* base;
  size_t off = 0;
  explicit Bump(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

int check_dims(const dflash_dims& d, const char* who) {
  DF_CHECK(d.dtype == DFLASH_F32 || d.dtype == DFLASH_BF16, "%s: dtype %d not F32/BF16", who, d.dtype);
  DF_CHECK(d.hidden > 0 && d.hidden % 8 == 0, "%s: hidden %d must be a positive multiple of 8", who, d.hidden);
  DF_CHECK(d.head_dim == 64 || d.head_dim == 128, "%s: head_dim %d must be 64 or 128", who, d.head_dim);
  DF_CHECK(d.n_q_heads > 0 && d.n_kv_heads > 0 && d.n_q_heads % d.n_kv_heads == 0,
           "%s: n_q_heads %d must be a positive multiple of n_kv_heads %d", who, d.n_q_heads, d.n_kv_heads);
  DF_CHECK(d.intermediate > 0 && d.intermediate % 8 == 0, "%s: intermediate %d must be a multiple of 8", who,
           d.intermediate);
  DF_CHECK((d.n_q_heads * d.head_dim) % 8 == 0, "%s: n_q_heads*head_dim must be a multiple of 8", who);
  DF_CHECK(d.vocab > 0, "%s: vocab must be positive", who);
  DF_CHECK(d.rms_eps >= 0.f && d.rope_theta > 0.f, "%s: rms_eps >= 0 and rope_theta > 0 required", who);
  return DFLASH_OK;
}

struct Ctx {
  uint32_t* status;
  uint32_t* counters;
};

Ctx header(void* ws) {
  Ctx c;
  c.status = static_cast<uint32_t*>(ws);
  c.counters = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + kHeaderBytes);
  return c;
}

// ------------------------------------------------------------------ GEMMs

size_t gemm_scratch_bytes(const GemmDesc& g, int sms) {
  return g.dtype == DFLASH_BF16 && gemm_tc_supported(g) ? gemm_tc_workspace(g, sms) : 0;
}

// Algorithmic bytes of a GEMM launch: every weight row once, the token rows
// once, the outputs once (residual outputs read and written).
double gemm_bytes(const GemmDesc& g) {
  const double es = g.dtype == DFLASH_BF16 ? 2.0 : 4.0;
  const double rows = (double)g.nseg * g.seg_rows;
  double b = rows * g.K * es + (double)g.M * g.K * es;
  if (g.kind == EPI_RESID) b += 2.0 * g.M * rows * 4.0;
  else if (g.kind == EPI_STORE) b += (double)g.M * rows * 4.0;
  else if (g.kind == EPI_SWIGLU) b += (double)g.M * g.inter * es;
  else b += (double)g.M * rows * es;
  return b;
}

cudaError_t run_gemm(const GemmDesc& g, void* gpart, size_t gpart_bytes, const Ctx& c, int sms,
                     cudaStream_t st) {
  const bool tc = g.dtype == DFLASH_BF16 && gemm_tc_supported(g);
  trace_pre(st, tc ? TF_GEMM_TC : TF_GEMM_SIMT);
  cudaError_t e = tc ? launch_gemm_tc(g, gpart, gpart_bytes, c.counters, c.status, sms, st)
                     : launch_gemm_simt(g, st);
  trace_post(st, gemm_bytes(g));
  return e;
}

GemmDesc gemm_base(int dtype, int M, int K, const void* X, const int32_t* base_pos, const int32_t* valid,
                   int rows) {
  GemmDesc g;
  memset(&g, 0, sizeof(g));
  g.dtype = dtype;
  g.M = M;
  g.K = K;
  g.X = X;
  g.nseg = 1;
  g.base_pos = base_pos;
  g.valid = valid;
  g.rows = rows;
  return g;
}

// ----------------------------------------------------------- decoder layer

struct LayerScratch {
  void *x, *x2, *q, *kb, *vb, *attn, *act;  // x: attention input, x2: MLP input (the same buffer by default)
  float* apart;
  void* gpart;
  size_t gpart_bytes;
  // DFlash 2 convolutions (draft layers with conv_rank > 0)
  void* xc;    // [M][H] convolved projection input
  float* yc;   // [M][H] sublayer output before its convolution
  float* zc;   // [M][r] tap generator activations
};

// The four convolutions of one draft layer (w1 [4][r][H], w2 [4][2H][r]).
struct LayerConv {
  const void* w1;
  const void* w2;
  int r;
};

struct LayerShape {
  dflash_dims d;
  int S, rows, mode, max_pos, cap, window;
};

void layer_gemms(const LayerShape& L, const dflash_layer_weights* w, GemmDesc* g4) {
  const dflash_dims& d = L.d;
  const int M = L.S * L.rows, H = d.hidden, QD = d.n_q_heads * d.head_dim, KD = d.n_kv_heads * d.head_dim;
  GemmDesc qkv = gemm_base(d.dtype, M, H, nullptr, nullptr, nullptr, L.rows);
  qkv.seg_w[0] = w ? w->w_qkv : nullptr;
  qkv.seg_rows = QD + 2 * KD;
  qkv.kind = EPI_QKV;
  qkv.nq = d.n_q_heads;
  qkv.nkv = d.n_kv_heads;
  qkv.d = d.head_dim;
  GemmDesc o = gemm_base(d.dtype, M, QD, nullptr, nullptr, nullptr, L.rows);
  o.seg_w[0] = w ? w->w_o : nullptr;
  o.seg_rows = H;
  o.kind = EPI_RESID;
  o.ldo = H;
  GemmDesc gu = gemm_base(d.dtype, M, H, nullptr, nullptr, nullptr, L.rows);
  gu.seg_w[0] = w ? w->w_gu : nullptr;
  gu.seg_rows = 2 * d.intermediate;
  gu.kind = EPI_SWIGLU;
  gu.inter = d.intermediate;
  GemmDesc dn = gemm_base(d.dtype, M, d.intermediate, nullptr, nullptr, nullptr, L.rows);
  dn.seg_w[0] = w ? w->w_down : nullptr;
  dn.seg_rows = H;
  dn.kind = EPI_RESID;
  dn.ldo = H;
  g4[0] = qkv;
  g4[1] = o;
  g4[2] = gu;
  g4[3] = dn;
}

AttnDesc attn_shape(const LayerShape& L) {
  AttnDesc a;
  memset(&a, 0, sizeof(a));
  a.dtype = L.d.dtype;
  a.mode = L.mode;
  a.n_seqs = L.S;
  a.rows = L.rows;
  a.nq = L.d.n_q_heads;
  a.nkv = L.d.n_kv_heads;
  a.d = L.d.head_dim;
  a.cap = L.cap;
  a.window = L.window;
  a.max_pos = L.max_pos;
  return a;
}

void carve_layer(Bump& b, const LayerShape& L, int sms, LayerScratch& s, int conv_rank = 0) {
  const dflash_dims& d = L.d;
  const size_t es = elem_size(d.dtype);
  const size_t M = (size_t)L.S * L.rows;
  const size_t QD = (size_t)d.n_q_heads * d.head_dim;
  s.x = b.take(M * d.hidden * es);
  s.x2 = s.x;
  s.q = b.take(M * QD * es);
  s.kb = b.take((size_t)L.S * d.n_kv_heads * L.rows * d.head_dim * es);
  s.vb = b.take((size_t)L.S * d.n_kv_heads * L.rows * d.head_dim * es);
  s.attn = b.take(M * QD * es);
  s.act = b.take(M * d.intermediate * es);
  s.apart = static_cast<float*>(b.take(attn_workspace(attn_shape(L))));
  GemmDesc g4[4];
  layer_gemms(L, nullptr, g4);
  size_t gp = 0;
  for (auto& g : g4) gp = std::max(gp, gemm_scratch_bytes(g, sms));
  s.gpart_bytes = gp;
  s.gpart = b.take(gp);
  s.xc = nullptr;
  s.yc = nullptr;
  s.zc = nullptr;
  if (conv_rank > 0) {
    s.xc = b.take(M * d.hidden * es);
    s.yc = static_cast<float*>(b.take(M * d.hidden * sizeof(float)));
    s.zc = static_cast<float*>(b.take(M * (size_t)conv_rank * sizeof(float)));
  }
}

// Convolution `at` (0 attention input, 1 attention output, 2 MLP input, 3 MLP
// output) of a draft layer over the M rows of u.
static cudaError_t layer_conv(const LayerShape& L, const LayerConv& cv, int at, const void* u, void* out, int resid,
                              const LayerScratch& s, cudaStream_t st) {
  const dflash_dims& d = L.d;
  const size_t es = elem_size(d.dtype);
  ConvDesc c;
  c.dtype = d.dtype;
  c.M = L.S * L.rows;
  c.H = d.hidden;
  c.r = cv.r;
  c.rows = L.rows;
  c.w1 = static_cast<const char*>(cv.w1) + (size_t)at * cv.r * d.hidden * es;
  c.w2 = static_cast<const char*>(cv.w2) + (size_t)at * 2 * d.hidden * cv.r * es;
  c.u = u;
  c.out = out;
  c.resid = resid;
  c.z = s.zc;
  return launch_dyn_conv(c, st);
}

static double conv_bytes(const LayerShape& L, const LayerConv& cv) {
  const double es = elem_size(L.d.dtype), M = (double)L.S * L.rows, H = L.d.hidden;
  return 3.0 * cv.r * H * es + 2.0 * M * H * 4.0;
}

int check_layer_shape(const LayerShape& L, const char* who) {
  DF_CHECK(L.S > 0 && L.rows > 0, "%s: n_seqs and rows must be positive", who);
  DF_CHECK(L.mode == DFLASH_ATTN_CAUSAL || L.mode == DFLASH_ATTN_BLOCK_BIDIR, "%s: bad attn_mode", who);
  DF_CHECK(L.cap > 0, "%s: kv capacity must be positive", who);
  DF_CHECK(L.max_pos >= L.rows, "%s: max_pos must cover base_pos + rows", who);
  if (L.mode == DFLASH_ATTN_CAUSAL) {
    DF_CHECK(L.window == 0, "%s: causal layers take no window", who);
    DF_CHECK(L.max_pos <= L.cap, "%s: max_pos %d exceeds cache capacity %d", who, L.max_pos, L.cap);
  } else {
    DF_CHECK(L.window == 0 ? L.max_pos - L.rows <= L.cap : L.window == L.cap,
             "%s: context cache too small (window ring needs capacity == window)", who);
  }
  if (L.mode == DFLASH_ATTN_BLOCK_BIDIR)
    DF_CHECK(L.rows <= 64, "%s: a bidirectional block holds at most 64 rows", who);
  AttnDesc a = attn_shape(L);
  const int grp = L.d.n_q_heads / L.d.n_kv_heads;
  const int n_qt = (L.rows * grp + 63) / 64;
  DF_CHECK((long)L.S * L.d.n_kv_heads * n_qt <= 16384, "%s: too many attention groups (n_seqs*n_kv*tiles > 16384)",
           who);
  (void)a;
  return DFLASH_OK;
}

// The shared fields of a page scatter (the per-layer pointers are the caller's).
static KvScatter kv_scatter_base(const dflash_dims& d, int S, int rows, const int32_t* base_pos, const int32_t* valid,
                                 int window, int cap, int rope_max_pos, const dflash_kv& kv, const Ctx& c) {
  KvScatter k;
  memset(&k, 0, sizeof(k));
  k.dtype = d.dtype;
  k.n_layers = 1;
  k.S = S;
  k.rows = rows;
  k.nkv = d.n_kv_heads;
  k.d = d.head_dim;
  k.base_pos = base_pos;
  k.valid = valid;
  k.window = window;
  k.cap = cap;
  k.rope_max_pos = rope_max_pos;
  k.ps = kv.page_size;
  k.max_pages = kv.max_pages;
  k.pool = kv.pool_pages;
  k.status = c.status;
  return k;
}

int run_layer(const LayerShape& L, const dflash_layer_weights& w, const dflash_kv& kv, float* h,
              const int32_t* base_pos, const float* rope_cs, int rope_max_pos, void* tap, int tap_stride, int tap_offset,
              const LayerScratch& s, const Ctx& c, int sms, cudaStream_t st, const LayerConv* cv = nullptr) {
  const dflash_dims& d = L.d;
  const int M = L.S * L.rows, H = d.hidden;
  GemmDesc g4[4];
  layer_gemms(L, &w, g4);
  for (auto& g : g4) g.base_pos = base_pos;
  const bool causal = L.mode == DFLASH_ATTN_CAUSAL;

  DF_LAUNCH(st, TF_RMSNORM, 0, launch_rmsnorm(d.dtype, h, w.ln1, M, H, d.rms_eps, s.x, st));
  if (cv) DF_LAUNCH(st, TF_CONV, conv_bytes(L, *cv), layer_conv(L, *cv, 0, s.x, s.xc, 0, s, st));
  GemmDesc& qkv = g4[0];
  qkv.X = cv ? s.xc : s.x;
  qkv.q_out = s.q;
  // Causal rows go straight to their cache slots; bidirectional block rows
  // and the rows of a paged cache go to the block scratch (a paged cache
  // receives them from the page scatter below).
  const bool direct = causal && kv.pages == nullptr;
  qkv.k_dst[0] = direct ? kv.k : s.kb;
  qkv.v_dst[0] = direct ? kv.v : s.vb;
  qkv.kv_cap = direct ? kv.capacity : L.rows;
  qkv.kv_window = 0;
  qkv.kv_slot_mode = direct ? 1 : 0;
  qkv.rope_cs = rope_cs;
  qkv.rope_max_pos = rope_max_pos;
  DF_CUDA(run_gemm(qkv, s.gpart, s.gpart_bytes, c, sms, st));
  if (causal && kv.pages) {
    KvScatter ks = kv_scatter_base(L.d, L.S, L.rows, base_pos, nullptr, 0, kv.capacity, rope_max_pos, kv, c);
    ks.kb[0] = s.kb;
    ks.vb[0] = s.vb;
    ks.kpool[0] = kv.k;
    ks.vpool[0] = kv.v;
    ks.pages[0] = kv.pages;
    DF_LAUNCH(st, TF_PAGE, 0, launch_kv_page_scatter(ks, st));
  }

  AttnDesc a = attn_shape(L);
  a.base_pos = base_pos;
  a.q = s.q;
  a.kc = kv.k;
  a.vc = kv.v;
  a.pages = kv.pages;
  a.ps = kv.page_size;
  a.max_pages = kv.max_pages;
  a.pool = kv.pool_pages;
  a.kb = s.kb;
  a.vb = s.vb;
  a.out = s.attn;
  a.partials = s.apart;
  a.counters = c.counters;
  a.status = c.status;
  DF_LAUNCH(st, TF_ATTN, 0, launch_attention(a, st));

  // With convolutions the O and down projections store their output, which
  // the convolution then adds to the residual.
  GemmDesc& o = g4[1];
  o.X = s.attn;
  o.out_f32 = cv ? s.yc : h;
  if (cv) o.kind = EPI_STORE;
  DF_CUDA(run_gemm(o, s.gpart, s.gpart_bytes, c, sms, st));
  if (cv) DF_LAUNCH(st, TF_CONV, conv_bytes(L, *cv), layer_conv(L, *cv, 1, s.yc, h, 1, s, st));

  DF_LAUNCH(st, TF_RMSNORM, 0, launch_rmsnorm(d.dtype, h, w.ln2, M, H, d.rms_eps, s.x2, st));
  if (cv) DF_LAUNCH(st, TF_CONV, conv_bytes(L, *cv), layer_conv(L, *cv, 2, s.x2, s.xc, 0, s, st));
  GemmDesc& gu = g4[2];
  gu.X = cv ? s.xc : s.x2;
  gu.act_out = s.act;
  DF_CUDA(run_gemm(gu, s.gpart, s.gpart_bytes, c, sms, st));

  GemmDesc& dn = g4[3];
  dn.X = s.act;
  dn.out_f32 = cv ? s.yc : h;
  if (cv) dn.kind = EPI_STORE;
  DF_CUDA(run_gemm(dn, s.gpart, s.gpart_bytes, c, sms, st));
  if (cv) DF_LAUNCH(st, TF_CONV, conv_bytes(L, *cv), layer_conv(L, *cv, 3, s.yc, h, 1, s, st));

  if (tap) DF_LAUNCH(st, TF_TAP, 0, launch_store_tap(d.dtype, h, M, H, tap, tap_stride, tap_offset, st));
  return DFLASH_OK;
}

int check_ws(void* ws, size_t ws_bytes, size_t need, const char* who) {
  if (!ws) return fail(DFLASH_ERR_INVALID_ARG, "%s: workspace is NULL", who);
  if (ws_bytes < need)
    return fail(DFLASH_ERR_WORKSPACE, "%s: workspace %zu bytes, %zu required", who, ws_bytes, need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "%s: workspace must be 256-byte aligned", who);
  return DFLASH_OK;
}

// A paged cache: page size a multiple of the 128-key attention chunk,
// capacity == max_pages * page_size.
int check_kv_pages(const dflash_kv& kv, const char* who) {
  if (!kv.pages) return DFLASH_OK;
  DF_CHECK(kv.page_size > 0 && kv.page_size % 128 == 0, "%s: page_size must be a positive multiple of 128", who);
  DF_CHECK(kv.max_pages > 0 && kv.pool_pages > 0, "%s: max_pages and pool_pages must be positive", who);
  DF_CHECK((long)kv.max_pages * kv.page_size == kv.capacity, "%s: capacity must equal max_pages * page_size", who);
  DF_CHECK((long)kv.pool_pages * kv.page_size <= (1L << 30), "%s: page pool too large", who);
  return DFLASH_OK;
}

int check_weights(const dflash_layer_weights& w, const char* who) {
  DF_CHECK(w.w_qkv && w.w_o && w.w_gu && w.w_down && w.ln1 && w.ln2, "%s: null layer weight", who);
  return DFLASH_OK;
}

// --------------------------------------------------------------- LM head

// Algorithmic bytes of the LM head: every vocabulary row once + the token rows.
double head_bytes(const HeadDesc& h) {
  const double es = h.dtype == DFLASH_BF16 ? 2.0 : 4.0;
  return (double)h.V * h.H * es + (double)h.M * h.H * es;
}

// Sequences per LM-head launch: whole sequences, at most 256 token rows.
int head_seqs_per_launch(int block) { return block >= 256 ? 1 : 256 / block; }

HeadDesc head_shape(const dflash_dims& d, int S, int block, int mode) {
  HeadDesc h;
  memset(&h, 0, sizeof(h));
  h.dtype = d.dtype;
  h.M = S * block;
  h.H = d.hidden;
  h.V = d.vocab;
  h.n_seqs = S;
  h.block = block;
  h.mode = mode;
  return h;
}

// Measure or carve the whole draft call.
struct DraftScratch {
  float* h;
  LayerScratch ls;
  void* xf;
  void* hpart;
  int32_t* cand;
  float* proj;     // path selector projections (path_topk > 0)
  float* logits;   // draft logit rows when the CUDA-core head feeds the top-k merge
};

LayerShape draft_layer_shape(const dflash_draft_args* a, int j) {
  LayerShape L;
  L.d = a->dims;
  L.S = a->n_seqs;
  L.rows = a->block;
  L.mode = DFLASH_ATTN_BLOCK_BIDIR;
  L.max_pos = a->max_pos;
  L.cap = a->kv_layers[j].capacity;
  L.window = a->kv_layers[j].window;
  return L;
}

size_t carve_draft(Bump& b, const dflash_draft_args* a, int sms, DraftScratch& s) {
  const dflash_dims& d = a->dims;
  const size_t M = (size_t)a->n_seqs * a->block;
  b.take(kReservedBytes);
  s.h = static_cast<float*>(b.take(M * d.hidden * sizeof(float)));
  // layer scratch carved for the layer geometry that needs the most
  int jbest = 0;
  size_t bb = 0;
  for (int j = 0; j < a->n_layers; ++j) {
    Bump t(nullptr);
    LayerScratch tmp;
    carve_layer(t, draft_layer_shape(a, j), sms, tmp, a->conv_rank);
    if (t.off > bb) {
      bb = t.off;
      jbest = j;
    }
  }
  carve_layer(b, draft_layer_shape(a, jbest), sms, s.ls, a->conv_rank);
  s.xf = b.take(M * d.hidden * elem_size(d.dtype));
  HeadDesc hd = head_shape(d, a->n_seqs, a->block, a->path_topk > 0 ? 2 : 0);
  hd.topk = a->path_topk;
  hd.x = s.xf;
  s.hpart = b.take(head_workspace(hd, sms));
  s.cand = static_cast<int32_t*>(b.take((size_t)a->n_seqs * a->block * 16 * sizeof(int32_t)));
  s.proj = nullptr;
  s.logits = nullptr;
  if (a->path_topk > 0) {
    s.proj = static_cast<float*>(
        b.take(path_proj_floats(a->n_seqs, a->block, a->path_topk, a->path_rank) * sizeof(float)));
    HeadDesc one = hd;  // the shape of one head launch
    one.n_seqs = std::min(a->n_seqs, head_seqs_per_launch(a->block));
    one.M = one.n_seqs * a->block;
    if (!head_tc_supported(one) && a->logits == nullptr)
      s.logits = static_cast<float*>(b.take((size_t)a->n_seqs * (a->block - 1) * d.vocab * sizeof(float)));
  }
  return b.off;
}

// Sequences [s0, s0 + n) of an LM-head problem.
HeadDesc head_slice(const HeadDesc& h, int s0, int n) {
  HeadDesc c = h;
  const int B = h.block, Bd = B - 1;
  const bool verify = h.mode == 1;
  c.n_seqs = n;
  c.M = n * B;
  c.x = static_cast<const char*>(h.x) + (size_t)s0 * B * h.H * elem_size(h.dtype);
  if (h.drafts) c.drafts = h.drafts + (size_t)s0 * Bd;
  if (h.drafts_out) c.drafts_out = h.drafts_out + (size_t)s0 * Bd;
  if (h.argmax) c.argmax = h.argmax + (size_t)s0 * B;
  if (h.margin) c.margin = h.margin + (size_t)s0 * (verify ? B : Bd);
  if (h.accept_len) c.accept_len = h.accept_len + s0;
  if (h.out_tokens) c.out_tokens = h.out_tokens + (size_t)s0 * B;
  if (h.next_anchor) c.next_anchor = h.next_anchor + s0;
  if (h.base_pos) c.base_pos = h.base_pos + s0;
  if (h.commit_base) c.commit_base = h.commit_base + s0;
  if (h.commit_count) c.commit_count = h.commit_count + s0;
  if (h.cand_out) c.cand_out = h.cand_out + (size_t)s0 * Bd * h.topk;
  if (h.logits) c.logits = h.logits + (size_t)s0 * (verify ? B : Bd) * h.V;
  return c;
}

// The LM head in launches of whole sequences (at most 256 token rows each);
// in top-k mode each launch's candidates are merged after it.
int run_head(const HeadDesc& h, int sms, cudaStream_t st) {
  const int per = head_seqs_per_launch(h.block);
  for (int s0 = 0; s0 < h.n_seqs; s0 += per) {
    const HeadDesc c = head_slice(h, s0, std::min(per, h.n_seqs - s0));
    DF_LAUNCH(st, TF_HEAD, head_bytes(c), launch_head(c, sms, st));
    if (c.topk > 0) {
      int n_tiles = 0;
      const void* tl = head_tc_supported(c) ? head_tc_tlist(c, sms, &n_tiles) : nullptr;
      DF_LAUNCH(st, TF_PATH, 0, launch_topk_merge(c, tl, n_tiles, st));
    }
  }
  return DFLASH_OK;
}

}  // namespace

static int check_verify_shape(const dflash_verify_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  DF_CHECK(a->n_seqs > 0 && a->block >= 1, "%s: n_seqs > 0 and block >= 1 required", who);
  DF_CHECK((long)a->n_seqs * a->block <= 1024, "%s: n_seqs*block must be <= 1024", who);
  return DFLASH_OK;
}


namespace dfl {
// Sets the thread-local error text from another translation unit.
int abi_fail(int code, const char* msg) { return fail(code, "%s", msg); }

// Every host-side check of dflash_verify_accept (shapes, then pointers).
int verify_check(const dflash_verify_args* a, const char* who) {
  int rc = check_verify_shape(a, who);
  if (rc) return rc;
  DF_CHECK(a->h && a->final_norm && a->lm_head && a->argmax && a->accept_len && a->out_tokens,
           "%s: NULL pointer", who);
  DF_CHECK(a->drafts || a->block == 1, "%s: drafts required when block > 1", who);
  DF_CHECK(!a->commit_base || a->base_pos, "%s: commit_base needs base_pos", who);
  return DFLASH_OK;
}
}  // namespace dfl

// =================================================================== ABI

extern "C" {

int32_t dflash_abi_version(void) { return DFLASH_ABI_VERSION; }

int32_t dflash_build_flags(void) {
#ifdef DFLASH_CHECKED
  return DFLASH_BUILD_CHECKED;
#else
  return 0;
#endif
}

const char* dflash_last_error(void) { return g_err; }

int dflash_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* cos_sin, dflash_stream_t stream) {
  DF_CHECK(cos_sin != nullptr, "dflash_rope_table: cos_sin is NULL");
  DF_CHECK(head_dim > 0 && head_dim % 2 == 0 && max_pos > 0 && theta > 0.f,
           "dflash_rope_table: need theta > 0, even head_dim > 0, max_pos > 0");
  DF_LAUNCH((cudaStream_t)stream, TF_ROPE, 0,
            launch_rope_table(theta, head_dim, max_pos, cos_sin, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_workspace_init(void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DF_CHECK(ws != nullptr && ws_bytes >= kReservedBytes, "dflash_workspace_init: workspace below %zu bytes",
           kReservedBytes);
  DF_CUDA(cudaMemsetAsync(ws, 0, kReservedBytes, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_workspace_control(void* ws, size_t ws_bytes, uint64_t wait_limit_ns, int32_t stall_kv_loads,
                             dflash_stream_t stream) {
  DF_CHECK(ws != nullptr && ws_bytes >= kReservedBytes, "dflash_workspace_control: workspace below %zu bytes",
           kReservedBytes);
  DF_CHECK((reinterpret_cast<uintptr_t>(ws) & 255) == 0, "dflash_workspace_control: workspace must be 256-byte aligned");
  DF_CHECK(stall_kv_loads >= 0 && stall_kv_loads <= 3, "dflash_workspace_control: stall switches are bits 0 and 1");
  // bytes 8..15: the wait limit, 16..19: the stall switches (see wait_limit_ns)
  uint32_t ctl[4] = {(uint32_t)(wait_limit_ns & 0xffffffffu), (uint32_t)(wait_limit_ns >> 32),
                     (uint32_t)stall_kv_loads, 0u};
  DF_CUDA(cudaMemcpyAsync(static_cast<char*>(ws) + 8, ctl, sizeof(ctl), cudaMemcpyHostToDevice,
                          (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_read_status(void* ws, dflash_stream_t stream, int32_t* host_status) {
  DF_CHECK(ws != nullptr && host_status != nullptr, "dflash_read_status: NULL argument");
  uint32_t v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  DF_CUDA(cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st));
  DF_CUDA(cudaStreamSynchronize(st));
  DF_CUDA(cudaMemsetAsync(ws, 0, sizeof(uint32_t), st));
  DF_CUDA(cudaStreamSynchronize(st));
  *host_status = (v & ST_NUMERIC)   ? DFLASH_ERR_NUMERIC
                 : (v & ST_TIMEOUT) ? DFLASH_ERR_TIMEOUT
                 : (v & ST_RANGE)   ? DFLASH_ERR_INVALID_ARG
                 : (v & ST_CHECK)   ? DFLASH_ERR_CHECK
                                    : DFLASH_OK;
  if (*host_status != DFLASH_OK) fail(*host_status, "device status word 0x%x", v);
  return DFLASH_OK;
}

// ----------------------------------------------------------------- embed

static int check_embed_shape(const dflash_embed_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  DF_CHECK(a->n_seqs >= 0 && a->rows > 0, "%s: bad n_seqs/rows", who);
  return DFLASH_OK;
}

int dflash_embed(const dflash_embed_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  int rc = check_embed_shape(a, "dflash_embed");
  if (rc) return rc;
  DF_CHECK(a->embed && a->first && a->h, "dflash_embed: NULL embed/first/h");
  DF_CHECK(a->rest != nullptr || (a->fill_token >= 0 && a->fill_token < a->dims.vocab),
           "dflash_embed: fill_token out of range");
  rc = check_ws(ws, ws_bytes, kReservedBytes, "dflash_embed");
  if (rc) return rc;
  DF_LAUNCH((cudaStream_t)stream, TF_EMBED, 0,
            launch_embed(a->dims.dtype, a->embed, a->dims.hidden, a->dims.vocab, a->n_seqs, a->rows, a->first,
                         a->rest, a->fill_token, a->h, header(ws).status, (cudaStream_t)stream));
  return DFLASH_OK;
}

// --------------------------------------------------------- decoder layer

static LayerShape layer_shape_of(const dflash_layer_args* a) {
  LayerShape L;
  L.d = a->dims;
  L.S = a->n_seqs;
  L.rows = a->rows;
  L.mode = a->attn_mode;
  L.max_pos = a->max_pos;
  L.cap = a->kv.capacity;
  L.window = a->kv.window;
  return L;
}

static size_t layer_ws(const dflash_layer_args* a, int sms) {
  Bump b(nullptr);
  b.take(kReservedBytes);
  LayerScratch s;
  carve_layer(b, layer_shape_of(a), sms, s);
  return b.off;
}

static int check_layer_args_shape(const dflash_layer_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  rc = check_kv_pages(a->kv, who);
  if (rc) return rc;
  return check_layer_shape(layer_shape_of(a), who);
}

int dflash_decoder_layer_forward(const dflash_layer_args* a, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream) {
  const char* who = "dflash_decoder_layer_forward";
  int rc = check_layer_args_shape(a, who);
  if (rc) return rc;
  rc = check_weights(a->w, who);
  if (rc) return rc;
  DF_CHECK(a->base_pos && a->h && a->kv.k && a->kv.v && a->rope_cs, "%s: NULL pointer", who);
  LayerShape L = layer_shape_of(a);
  DF_CHECK(a->max_pos <= a->rope_max_pos, "%s: max_pos %d beyond the RoPE table (%d)", who, a->max_pos,
           a->rope_max_pos);
  {
    const void* st[] = {a->out_x_attn, a->out_q, a->out_kb, a->out_vb, a->out_attn, a->out_x_mlp, a->out_act};
    for (const void* p : st)
      DF_CHECK((reinterpret_cast<uintptr_t>(p) & 15) == 0, "%s: stage outputs must be 16-byte aligned", who);
  }
  DF_CHECK(!a->tap || (a->tap_stride >= a->dims.hidden && a->tap_offset >= 0 &&
                        a->tap_offset + a->dims.hidden <= a->tap_stride),
           "%s: bad tap stride/offset", who);
  const int sms = num_sms();
  rc = check_ws(ws, ws_bytes, layer_ws(a, sms), who);
  if (rc) return rc;
  Bump b(ws);
  b.take(kReservedBytes);
  LayerScratch s;
  carve_layer(b, L, sms, s);
  // stage outputs replace the scratch they would have occupied
  if (a->out_x_attn) s.x = a->out_x_attn;
  if (a->out_x_mlp) s.x2 = a->out_x_mlp;
  if (a->out_q) s.q = a->out_q;
  if (a->out_kb && L.mode == DFLASH_ATTN_BLOCK_BIDIR) s.kb = a->out_kb;
  if (a->out_vb && L.mode == DFLASH_ATTN_BLOCK_BIDIR) s.vb = a->out_vb;
  if (a->out_attn) s.attn = a->out_attn;
  if (a->out_act) s.act = a->out_act;
  return run_layer(L, a->w, a->kv, a->h, a->base_pos, a->rope_cs, a->rope_max_pos, a->tap, a->tap_stride, a->tap_offset, s,
                   header(ws), sms, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- fusion

static size_t fuse_ws(const dflash_fuse_args* a, int sms, float** z, void** cbuf, void** gpart, size_t* gp,
                      char* base, void** kscr = nullptr, void** vscr = nullptr) {
  const dflash_dims& d = a->dims;
  const size_t M = (size_t)a->n_seqs * a->rows;
  Bump b(base);
  b.take(kReservedBytes);
  *z = static_cast<float*>(b.take(M * d.hidden * sizeof(float)));
  *cbuf = b.take(M * d.hidden * elem_size(d.dtype));
  GemmDesc fc = gemm_base(d.dtype, (int)M, a->n_taps * d.hidden, nullptr, nullptr, nullptr, a->rows);
  fc.seg_rows = d.hidden;
  fc.kind = EPI_STORE;
  GemmDesc kv = gemm_base(d.dtype, (int)M, d.hidden, nullptr, nullptr, nullptr, a->rows);
  kv.nseg = a->n_layers;
  kv.seg_row0 = d.n_q_heads * d.head_dim;
  kv.seg_rows = 2 * d.n_kv_heads * d.head_dim;
  kv.kind = EPI_QKV;
  kv.nq = d.n_q_heads;
  kv.nkv = d.n_kv_heads;
  kv.d = d.head_dim;
  *gp = std::max(gemm_scratch_bytes(fc, sms), gemm_scratch_bytes(kv, sms));
  *gpart = b.take(*gp);
  if (a->kv_layers[0].pages) {  // block scratch per layer for the page scatter
    const size_t blk = M * d.n_kv_heads * d.head_dim * elem_size(d.dtype);
    for (int j = 0; j < a->n_layers; ++j) {
      void* k = b.take(blk);
      void* v = b.take(blk);
      if (kscr) kscr[j] = k;
      if (vscr) vscr[j] = v;
    }
  }
  return b.off;
}

static int check_fuse_shape(const dflash_fuse_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  DF_CHECK(a->n_taps > 0 && a->n_taps <= 16, "%s: n_taps must be in [1, 16]", who);
  DF_CHECK(a->n_layers > 0 && a->n_layers <= DFLASH_MAX_LAYERS, "%s: n_layers must be in [1, %d]", who,
           DFLASH_MAX_LAYERS);
  DF_CHECK(a->n_seqs > 0 && a->rows > 0, "%s: n_seqs and rows must be positive", who);
  const int cap = a->kv_layers[0].capacity, win = a->kv_layers[0].window;
  for (int j = 0; j < a->n_layers; ++j) {
    const int rc2 = check_kv_pages(a->kv_layers[j], who);
    if (rc2) return rc2;
    DF_CHECK((a->kv_layers[j].pages == nullptr) == (a->kv_layers[0].pages == nullptr) &&
                 a->kv_layers[j].page_size == a->kv_layers[0].page_size &&
                 a->kv_layers[j].max_pages == a->kv_layers[0].max_pages &&
                 a->kv_layers[j].pool_pages == a->kv_layers[0].pool_pages,
             "%s: every layer's context cache must share its paging geometry", who);
    DF_CHECK(a->kv_layers[j].capacity == cap && a->kv_layers[j].window == win,
             "%s: every layer's context cache must share capacity and window", who);
  }
  DF_CHECK(cap > 0 && (win == 0 || win == cap), "%s: window ring needs capacity == window", who);
  return DFLASH_OK;
}

int dflash_fuse_context(const dflash_fuse_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_fuse_context";
  int rc = check_fuse_shape(a, who);
  if (rc) return rc;
  const dflash_dims& d = a->dims;
  DF_CHECK(a->w_fc && a->fc_norm && a->feats && a->base_pos && a->rope_cs, "%s: NULL pointer", who);
  for (int j = 0; j < a->n_layers; ++j)
    DF_CHECK(a->w_qkv_layers[j] && a->kv_layers[j].k && a->kv_layers[j].v, "%s: NULL layer %d pointer", who, j);
  const int cap = a->kv_layers[0].capacity, win = a->kv_layers[0].window;
  const int sms = num_sms();
  float* z;
  void *cbuf, *gpart;
  size_t gp;
  rc = check_ws(ws, ws_bytes, fuse_ws(a, sms, &z, &cbuf, &gpart, &gp, nullptr), who);
  if (rc) return rc;
  void* kscr[DFLASH_MAX_LAYERS] = {};
  void* vscr[DFLASH_MAX_LAYERS] = {};
  fuse_ws(a, sms, &z, &cbuf, &gpart, &gp, static_cast<char*>(ws), kscr, vscr);
  Ctx c = header(ws);
  cudaStream_t st = (cudaStream_t)stream;
  const int M = a->n_seqs * a->rows;

  GemmDesc fc = gemm_base(d.dtype, M, a->n_taps * d.hidden, a->feats, a->base_pos, a->valid, a->rows);
  fc.seg_w[0] = a->w_fc;
  fc.seg_rows = d.hidden;
  fc.kind = EPI_STORE;
  fc.out_f32 = z;
  fc.ldo = d.hidden;
  DF_CUDA(run_gemm(fc, gpart, gp, c, sms, st));
  DF_LAUNCH(st, TF_RMSNORM, 0, launch_rmsnorm(d.dtype, z, a->fc_norm, M, d.hidden, d.rms_eps, cbuf, st));
  if (a->c_out) DF_LAUNCH(st, TF_CONVERT, 0, launch_to_f32(d.dtype, cbuf, (size_t)M * d.hidden, a->c_out, st));

  GemmDesc kv = gemm_base(d.dtype, M, d.hidden, cbuf, a->base_pos, a->valid, a->rows);
  kv.nseg = a->n_layers;
  const bool paged = a->kv_layers[0].pages != nullptr;
  for (int j = 0; j < a->n_layers; ++j) {
    kv.seg_w[j] = a->w_qkv_layers[j];
    // a paged cache receives its rows from the page scatter below
    kv.k_dst[j] = paged ? kscr[j] : a->kv_layers[j].k;
    kv.v_dst[j] = paged ? vscr[j] : a->kv_layers[j].v;
  }
  kv.seg_row0 = d.n_q_heads * d.head_dim;
  kv.seg_rows = 2 * d.n_kv_heads * d.head_dim;
  kv.kind = EPI_QKV;
  kv.nq = d.n_q_heads;
  kv.nkv = d.n_kv_heads;
  kv.d = d.head_dim;
  kv.kv_cap = paged ? a->rows : cap;
  kv.kv_window = paged ? 0 : win;
  kv.kv_slot_mode = paged ? 0 : 1;
  kv.rope_cs = a->rope_cs;
  kv.rope_max_pos = a->rope_max_pos;
  DF_CUDA(run_gemm(kv, gpart, gp, c, sms, st));
  if (paged) {
    KvScatter ks = kv_scatter_base(d, a->n_seqs, a->rows, a->base_pos, a->valid, win, cap, a->rope_max_pos,
                                   a->kv_layers[0], c);
    ks.n_layers = a->n_layers;
    for (int j = 0; j < a->n_layers; ++j) {
      ks.kb[j] = kscr[j];
      ks.vb[j] = vscr[j];
      ks.kpool[j] = a->kv_layers[j].k;
      ks.vpool[j] = a->kv_layers[j].v;
      ks.pages[j] = a->kv_layers[j].pages;
    }
    DF_LAUNCH(st, TF_PAGE, 0, launch_kv_page_scatter(ks, st));
  }
  return DFLASH_OK;
}

// ----------------------------------------------------------------- draft

// One draft forward over the embedded block in s.h: every draft layer, the
// final norm, the fused LM head (argmax, or top-k candidates + path walk).
static int draft_round(const dflash_draft_args* a, const DraftScratch& s, const Ctx& c, int sms, cudaStream_t st) {
  const dflash_dims& d = a->dims;
  const int M = a->n_seqs * a->block;
  int rc;
  for (int j = 0; j < a->n_layers; ++j) {
    const LayerConv cv = {a->conv_rank > 0 ? a->conv_w1[j] : nullptr, a->conv_rank > 0 ? a->conv_w2[j] : nullptr,
                          a->conv_rank};
    rc = run_layer(draft_layer_shape(a, j), a->layers[j], a->kv_layers[j], s.h, a->base_pos, a->rope_cs,
                   a->rope_max_pos, nullptr, 0, 0, s.ls, c, sms, st, a->conv_rank > 0 ? &cv : nullptr);
    if (rc) return rc;
  }
  DF_LAUNCH(st, TF_RMSNORM, 0, launch_rmsnorm(d.dtype, s.h, a->final_norm, M, d.hidden, d.rms_eps, s.xf, st));
  HeadDesc h = head_shape(d, a->n_seqs, a->block, a->path_topk > 0 ? 2 : 0);
  h.topk = a->path_topk;
  h.x = s.xf;
  h.w = a->lm_head;
  h.drafts_out = a->drafts;
  h.cand_out = s.cand;
  h.logits = a->logits ? a->logits : s.logits;
  h.partials = static_cast<float*>(s.hpart);
  h.counters = c.counters;
  h.status = c.status;
  rc = run_head(h, sms, st);  // top-k mode: also each row's candidates, ranked by draft logit
  if (rc) return rc;
  if (a->path_topk > 0) {
    PathDesc p;
    memset(&p, 0, sizeof(p));
    p.dtype = d.dtype;
    p.n_seqs = a->n_seqs;
    p.block = a->block;
    p.topk = a->path_topk;
    p.rank = a->path_rank;
    p.H = d.hidden;
    p.V = d.vocab;
    p.embed = a->embed;
    p.u = a->path_u;
    p.v = a->path_v;
    p.anchor = a->anchor;
    p.cand = s.cand;
    p.path = a->drafts;
    p.proj = s.proj;
    p.status = c.status;
    p.T = a->path_temperature;
    p.seed = a->path_seed;
    p.cycle = a->path_cycle;
    p.base_pos = a->base_pos;
    p.logq = a->path_logq;
    p.cand_out = a->path_cand_out;
    DF_LAUNCH(st, TF_PATH, 0, launch_path_select(p, st));
  }
  return DFLASH_OK;
}

static int check_draft_shape(const dflash_draft_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  const dflash_dims& d = a->dims;
  DF_CHECK(a->n_layers > 0 && a->n_layers <= DFLASH_MAX_LAYERS, "%s: n_layers must be in [1, %d]", who,
           DFLASH_MAX_LAYERS);
  DF_CHECK(a->block >= 2 && a->n_seqs > 0, "%s: block >= 2 and n_seqs > 0 required", who);
  DF_CHECK((long)a->n_seqs * a->block <= 1024, "%s: n_seqs*block must be <= 1024", who);
  DF_CHECK(a->mask_token >= 0 && a->mask_token < d.vocab, "%s: mask_token out of range", who);
  DF_CHECK(a->path_topk >= 0 && a->path_topk <= 16, "%s: path_topk must be in [0, 16]", who);
  DF_CHECK(a->path_temperature >= 0.f && a->path_temperature == a->path_temperature,
           "%s: path_temperature must be >= 0", who);
  DF_CHECK(a->denoise_rounds >= 0 && a->denoise_rounds <= DFLASH_MAX_DENOISE_ROUNDS,
           "%s: denoise_rounds must be in [0, %d]", who, DFLASH_MAX_DENOISE_ROUNDS);
  DF_CHECK(a->conv_rank >= 0 && a->conv_rank <= DFLASH_MAX_CONV_RANK, "%s: conv_rank must be in [0, %d]", who,
           DFLASH_MAX_CONV_RANK);
  if (a->conv_rank > 0)
    DF_CHECK(a->conv_rank % 8 == 0 && d.hidden % 8 == 0, "%s: convolutions need conv_rank %% 8 == 0 and hidden %% 8 == 0",
             who);
  if (a->path_topk > 0)
    DF_CHECK(a->path_rank > 0 && a->path_rank <= 256 && d.hidden % 8 == 0,
             "%s: the path selector needs 0 < path_rank <= 256 and hidden %% 8 == 0", who);
  for (int j = 0; j < a->n_layers; ++j) {
    rc = check_kv_pages(a->kv_layers[j], who);
    if (rc) return rc;
    rc = check_layer_shape(draft_layer_shape(a, j), who);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_draft_block(const dflash_draft_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_draft_block";
  int rc = check_draft_shape(a, who);
  if (rc) return rc;
  const dflash_dims& d = a->dims;
  DF_CHECK(a->final_norm && a->embed && a->lm_head && a->anchor && a->base_pos && a->drafts && a->rope_cs,
           "%s: NULL pointer", who);
  DF_CHECK(a->max_pos <= a->rope_max_pos, "%s: max_pos beyond the RoPE table", who);
  for (int j = 0; a->conv_rank > 0 && j < a->n_layers; ++j)
    DF_CHECK(a->conv_w1[j] && a->conv_w2[j], "%s: NULL convolution weights of layer %d", who, j);
  if (a->path_topk > 0) DF_CHECK(a->path_u && a->path_v, "%s: path selector needs path_u and path_v", who);
  for (int j = 0; j < a->n_layers; ++j) {
    rc = check_weights(a->layers[j], who);
    if (rc) return rc;
    DF_CHECK(a->kv_layers[j].k && a->kv_layers[j].v, "%s: NULL context cache %d", who, j);
  }
  const int sms = num_sms();
  DraftScratch s;
  Bump m(nullptr);
  size_t need = carve_draft(m, a, sms, s);
  rc = check_ws(ws, ws_bytes, need, who);
  if (rc) return rc;
  Bump b(ws);
  carve_draft(b, a, sms, s);
  Ctx c = header(ws);
  cudaStream_t st = (cudaStream_t)stream;

  // Round 1 embeds [anchor, mask, ...]; a later round embeds [anchor, the
  // drafts of the round before] (written to a->drafts by that round's head
  // or path walk, read here in stream order).
  const int rounds = a->denoise_rounds > 1 ? a->denoise_rounds : 1;
  for (int r = 0; r < rounds; ++r) {
    DF_LAUNCH(st, TF_EMBED, 0,
              launch_embed(d.dtype, a->embed, d.hidden, d.vocab, a->n_seqs, a->block, a->anchor,
                           r == 0 ? nullptr : a->drafts, a->mask_token, s.h, c.status, st));
    rc = draft_round(a, s, c, sms, st);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

// ---------------------------------------------------------------- verify

static size_t verify_ws(const dflash_verify_args* a, int sms, void** xf, void** hpart, char* base) {
  Bump b(base);
  b.take(kReservedBytes);
  const size_t M = (size_t)a->n_seqs * a->block;
  *xf = b.take(M * a->dims.hidden * elem_size(a->dims.dtype));
  *hpart = b.take(head_workspace(head_shape(a->dims, a->n_seqs, a->block, 1), sms));
  return b.off;
}

int dflash_verify_accept(const dflash_verify_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_verify_accept";
  int rc = dfl::verify_check(a, who);
  if (rc) return rc;
  const int sms = num_sms();
  void *xf, *hpart;
  rc = check_ws(ws, ws_bytes, verify_ws(a, sms, &xf, &hpart, nullptr), who);
  if (rc) return rc;
  verify_ws(a, sms, &xf, &hpart, static_cast<char*>(ws));
  Ctx c = header(ws);
  cudaStream_t st = (cudaStream_t)stream;
  const dflash_dims& d = a->dims;
  const int M = a->n_seqs * a->block;
  DF_LAUNCH(st, TF_RMSNORM, 0, launch_rmsnorm(d.dtype, a->h, a->final_norm, M, d.hidden, d.rms_eps, xf, st));
  HeadDesc h = head_shape(d, a->n_seqs, a->block, 1);
  h.x = xf;
  h.w = a->lm_head;
  h.drafts = a->drafts;
  h.argmax = a->argmax;
  h.margin = a->margin;
  h.accept_len = a->accept_len;
  h.out_tokens = a->out_tokens;
  h.next_anchor = a->next_anchor;
  h.base_pos = a->base_pos;
  h.commit_base = a->commit_base;
  h.commit_count = a->commit_count;
  h.logits = a->logits;
  h.partials = static_cast<float*>(hpart);
  h.counters = c.counters;
  h.status = c.status;
  rc = run_head(h, sms, st);
  if (rc) return rc;
  return DFLASH_OK;
}

// ----------------------------------------------------------- path select

static size_t path_ws(const dflash_path_args* a) {
  return kReservedBytes + path_proj_floats(a->n_seqs, a->block, a->topk, a->rank) * sizeof(float);
}

static int check_path_shape(const dflash_path_args* a, const char* who) {
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_dims(a->dims, who);
  if (rc) return rc;
  DF_CHECK(a->n_seqs > 0 && a->block >= 2 && a->topk > 0 && a->topk <= 16 && a->rank > 0 && a->rank <= 256,
           "%s: need n_seqs > 0, block >= 2, 0 < topk <= 16, 0 < rank <= 256", who);
  DF_CHECK(a->dims.hidden % 8 == 0, "%s: hidden %% 8 == 0 required", who);
  return DFLASH_OK;
}

int dflash_path_select(const dflash_path_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_path_select";
  int rc = check_path_shape(a, who);
  if (rc) return rc;
  DF_CHECK(a->embed && a->path_u && a->path_v && a->anchor && a->cand && a->path, "%s: NULL pointer", who);
  DF_CHECK(a->temperature >= 0.f && a->temperature == a->temperature, "%s: temperature must be >= 0", who);
  DF_CHECK(a->temperature == 0.f || a->base_pos, "%s: the sampled walk needs base_pos", who);
  rc = check_ws(ws, ws_bytes, path_ws(a), who);
  if (rc) return rc;
  Ctx c = header(ws);
  PathDesc p;
  memset(&p, 0, sizeof(p));
  p.dtype = a->dims.dtype;
  p.n_seqs = a->n_seqs;
  p.block = a->block;
  p.topk = a->topk;
  p.rank = a->rank;
  p.H = a->dims.hidden;
  p.embed = a->embed;
  p.u = a->path_u;
  p.v = a->path_v;
  p.anchor = a->anchor;
  p.V = a->dims.vocab;
  p.cand = a->cand;
  p.path = a->path;
  p.margin = a->margin;
  p.proj = reinterpret_cast<float*>(static_cast<char*>(ws) + kReservedBytes);
  p.status = c.status;
  p.T = a->temperature;
  p.seed = a->seed;
  p.cycle = a->cycle;
  p.base_pos = a->base_pos;
  p.logq = a->logq;
  DF_LAUNCH((cudaStream_t)stream, TF_PATH, 0, launch_path_select(p, (cudaStream_t)stream));
  return DFLASH_OK;
}

// ------------------------------------------------------------- sampling

static size_t sample_ws(int S, int B, size_t* lse_off, size_t* k_off, size_t* part_off, size_t* filt_off = nullptr) {
  size_t off = kReservedBytes;
  *lse_off = off;
  off += ((size_t)S * B * sizeof(float) + 255) & ~size_t(255);
  *k_off = off;
  off += ((size_t)S * sizeof(int32_t) + 255) & ~size_t(255);
  *part_off = off;
  off += sample_part_bytes(S * B);
  if (filt_off) *filt_off = off;  // target rows' then draft rows' kept sets
  off += ((size_t)S * (2 * B - 1) * sizeof(RowFilter) + 255) & ~size_t(255);
  return off;
}

static int check_sample_shape(const dflash_dims& d, int S, int B, float T, int top_k, float top_p, const char* who) {
  DF_CHECK(d.vocab > 0 && d.vocab < (1 << 24), "%s: vocab must be in [1, 2^24)", who);
  DF_CHECK(top_k >= 0 && top_p >= 0.f && top_p <= 1.f, "%s: top_k >= 0 and 0 <= top_p <= 1 required", who);
  DF_CHECK(S > 0 && B >= 2 && (long)S * B <= 1024, "%s: n_seqs > 0, block >= 2, n_seqs*block <= 1024", who);
  DF_CHECK(T > 0.f && T == T, "%s: temperature must be > 0", who);
  return DFLASH_OK;
}

int dflash_sample_drafts(const dflash_sample_drafts_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_sample_drafts";
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_sample_shape(a->dims, a->n_seqs, a->block, a->temperature, a->top_k, a->top_p, who);
  if (rc) return rc;
  DF_CHECK(a->base_pos && a->draft_logits && a->drafts && a->draft_lse, "%s: NULL pointer", who);
  size_t lo, ko, po, fo;
  rc = check_ws(ws, ws_bytes, sample_ws(a->n_seqs, a->block, &lo, &ko, &po, &fo), who);
  if (rc) return rc;
  Ctx c = header(ws);
  SampleDesc d;
  memset(&d, 0, sizeof(d));
  d.n_seqs = a->n_seqs;
  d.block = a->block;
  d.V = a->dims.vocab;
  d.cycle = a->cycle;
  d.T = a->temperature;
  d.seed = a->seed;
  d.base_pos = const_cast<int32_t*>(a->base_pos);
  d.draft_logits = a->draft_logits;
  d.draft_lse_out = a->draft_lse;
  d.drafts_out = a->drafts;
  d.top_k = a->top_k;
  d.top_p = a->top_p;
  d.filt_d_out = reinterpret_cast<RowFilter*>(static_cast<char*>(ws) + fo) + (size_t)a->n_seqs * a->block;
  d.part = static_cast<char*>(ws) + po;
  d.counters = c.counters + kCtrSample;
  d.status = c.status;
  DF_LAUNCH((cudaStream_t)stream, TF_SAMPLE, 0, launch_sample_drafts(d, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_sample_accept(const dflash_sample_accept_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  const char* who = "dflash_sample_accept";
  DF_CHECK(a != nullptr, "%s: NULL args", who);
  int rc = check_sample_shape(a->dims, a->n_seqs, a->block, a->temperature, a->top_k, a->top_p, who);
  if (rc) return rc;
  DF_CHECK(a->target_logits && (a->draft_cand || (a->draft_logits && a->draft_lse)) && a->drafts && a->base_pos &&
               a->accept_len &&
               a->out_tokens,
           "%s: NULL pointer", who);
  DF_CHECK(!a->commit_base || a->update_base_pos, "%s: commit_base needs update_base_pos", who);
  DF_CHECK(!a->draft_cand || (a->draft_logq && a->draft_topk >= 1 && a->draft_topk <= 16),
           "%s: draft_cand needs draft_logq and 1 <= draft_topk <= 16", who);
  size_t lo, ko, po, fo;
  rc = check_ws(ws, ws_bytes, sample_ws(a->n_seqs, a->block, &lo, &ko, &po, &fo), who);
  if (rc) return rc;
  Ctx c = header(ws);
  SampleDesc d;
  memset(&d, 0, sizeof(d));
  d.n_seqs = a->n_seqs;
  d.block = a->block;
  d.V = a->dims.vocab;
  d.cycle = a->cycle;
  d.T = a->temperature;
  d.seed = a->seed;
  d.base_pos = a->base_pos;
  d.target_logits = a->target_logits;
  d.draft_logits = a->draft_logits;
  d.draft_lse = a->draft_lse;
  d.drafts = a->drafts;
  d.out_tokens = a->out_tokens;
  d.accept_len = a->accept_len;
  d.next_anchor = a->next_anchor;
  d.commit_base = a->commit_base;
  d.commit_count = a->commit_count;
  d.update_base = a->update_base_pos;
  if (a->draft_cand) {
    d.qk = a->draft_topk;
    d.qcand = a->draft_cand;
    d.qlogq = a->draft_logq;
  }
  d.top_k = a->top_k;
  d.top_p = a->top_p;
  if ((a->top_k > 0 && a->top_k < a->dims.vocab) || (a->top_p > 0.f && a->top_p < 1.f)) {
    RowFilter* f = reinterpret_cast<RowFilter*>(static_cast<char*>(ws) + fo);
    d.filt_t = f;
    d.filt_d = f + (size_t)a->n_seqs * a->block;
  }
  d.seq_k = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + ko);
  d.part = static_cast<char*>(ws) + po;
  d.counters = c.counters + kCtrSample;
  d.status = c.status;
  float* lse_t = reinterpret_cast<float*>(static_cast<char*>(ws) + lo);
  DF_LAUNCH((cudaStream_t)stream, TF_SAMPLE, 0, launch_sample_accept(d, lse_t, (cudaStream_t)stream));
  return DFLASH_OK;
}

// ------------------------------------------------------------- workspace

// The size of every op is computed only from arguments whose shape fields
// pass the op's checks (pointers are not needed to size a workspace); on a
// failed check the size is 0 and dflash_last_error() names the field.
size_t dflash_workspace_bytes(int32_t op, const void* args) {
  if (!args) {
    fail(DFLASH_ERR_INVALID_ARG, "dflash_workspace_bytes: NULL args");
    return 0;
  }
  const int sms = num_sms();
  const char* who = "dflash_workspace_bytes";
  switch (op) {
    case DFLASH_OP_EMBED:
      return check_embed_shape(static_cast<const dflash_embed_args*>(args), who) ? 0 : kReservedBytes;
    case DFLASH_OP_PATH: {
      const dflash_path_args* a = static_cast<const dflash_path_args*>(args);
      return check_path_shape(a, who) ? 0 : path_ws(a);
    }
    case DFLASH_OP_SAMPLE_DRAFTS: {
      const dflash_sample_drafts_args* a = static_cast<const dflash_sample_drafts_args*>(args);
      if (check_sample_shape(a->dims, a->n_seqs, a->block, a->temperature, a->top_k, a->top_p, who)) return 0;
      size_t lo, ko, po;
      return sample_ws(a->n_seqs, a->block, &lo, &ko, &po);
    }
    case DFLASH_OP_SAMPLE_ACCEPT: {
      const dflash_sample_accept_args* a = static_cast<const dflash_sample_accept_args*>(args);
      if (check_sample_shape(a->dims, a->n_seqs, a->block, a->temperature, a->top_k, a->top_p, who)) return 0;
      size_t lo, ko, po;
      return sample_ws(a->n_seqs, a->block, &lo, &ko, &po);
    }
    case DFLASH_OP_LAYER: {
      const dflash_layer_args* a = static_cast<const dflash_layer_args*>(args);
      return check_layer_args_shape(a, who) ? 0 : layer_ws(a, sms);
    }
    case DFLASH_OP_FUSE: {
      const dflash_fuse_args* a = static_cast<const dflash_fuse_args*>(args);
      if (check_fuse_shape(a, who)) return 0;
      float* z;
      void *cb, *gp;
      size_t g;
      return fuse_ws(a, sms, &z, &cb, &gp, &g, nullptr);
    }
    case DFLASH_OP_DRAFT: {
      const dflash_draft_args* a = static_cast<const dflash_draft_args*>(args);
      if (check_draft_shape(a, who)) return 0;
      DraftScratch s;
      Bump m(nullptr);
      return carve_draft(m, a, sms, s);
    }
    case DFLASH_OP_VERIFY: {
      const dflash_verify_args* a = static_cast<const dflash_verify_args*>(args);
      if (check_verify_shape(a, who)) return 0;
      void *xf, *hp;
      return verify_ws(a, sms, &xf, &hp, nullptr);
    }
    default:
      fail(DFLASH_ERR_INVALID_ARG, "dflash_workspace_bytes: unknown op %d", op);
      return 0;
  }
}

}  // extern "C"
