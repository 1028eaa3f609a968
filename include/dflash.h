/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash draft-and-verify library.
 *
 * One DFlash cycle ("DFlash: block-diffusion accelerated LLM speculative
 * decoding" guide, section 4 "how one task flows through the system"):
 *   1. context-feature fusion + KV injection      -> dflash_fuse_context
 *   2. single-step block-diffusion draft forward   -> dflash_draft_block
 *   3. causal target forward over the block        -> dflash_embed +
 *                                                     dflash_decoder_layer_forward (per layer)
 *   4. greedy verification + prefix acceptance     -> dflash_verify_accept
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers unless a field says "host".
 *    The caller owns every buffer (weights, caches, activations, outputs and
 *    the workspace); the library allocates no device memory and keeps no
 *    state beyond a thread-local error string and the opt-in, thread-local
 *    tracing state (dflash_trace_*).
 *  - Every call is asynchronous on the caller's `stream` and does no host
 *    synchronisation, except dflash_read_status.  Argument checks happen on
 *    the host before any launch; a failed check launches nothing.
 *  - Return value: DFLASH_OK (0) or a negative dflash_status.  On failure
 *    dflash_last_error() describes the cause.
 *  - Element type: dims.dtype selects bf16 or fp32 for weights, KV caches,
 *    tap features and the projection inputs; the residual stream `h` and
 *    logits are always fp32.
 *  - Weights are row-major [out][in].  A decoder layer's weights are
 *      w_qkv  [(n_q + 2 n_kv) * head_dim][hidden]   rows W_q, then W_k, then W_v
 *      w_o    [hidden][n_q * head_dim]
 *      w_gu   [2 * intermediate][hidden]            rows W_gate, then W_up
 *      w_down [hidden][intermediate]
 *      ln1, ln2 [hidden]                            RMSNorm gains
 *  - A KV cache of one layer is [n_seqs][n_kv][capacity][head_dim]; key
 *    vectors are stored already rotated (RoPE at their absolute position).
 *    Slots never written must hold finite values: zero-initialise caches.
 *  - A batch is n_seqs sequences of `rows` consecutive positions each: row i
 *    of sequence s sits at absolute position base_pos[s] + i and is row
 *    s*rows + i of every [M][...] activation (M = n_seqs * rows).
 *  - Workspace: every call takes (ws, ws_bytes).  Size it with
 *    dflash_workspace_bytes and zero it once with dflash_workspace_init; the
 *    library keeps it consistent afterwards.  Calls that share a workspace
 *    must be ordered on one stream.  Its first bytes hold the device status
 *    word that kernels raise on a numeric fault or an expired bounded wait.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_ABI_VERSION 8
#define DFLASH_MAX_LAYERS 16 /* draft layers handled by one fuse / draft call */

typedef struct CUstream_st* dflash_stream_t; /* == cudaStream_t */

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1, /* null pointer, bad size, inconsistent shapes */
  DFLASH_ERR_UNSUPPORTED = -2, /* shape/dtype/device the kernels do not cover */
  DFLASH_ERR_WORKSPACE = -3,   /* ws_bytes below dflash_workspace_bytes */
  DFLASH_ERR_CUDA = -4,        /* a CUDA runtime call failed */
  DFLASH_ERR_TIMEOUT = -5,     /* a bounded device wait gave up (status word) */
  DFLASH_ERR_NUMERIC = -6,     /* NaN reached an argmax (status word) */
  DFLASH_ERR_CHECK = -7        /* a device bounds assertion of the checked build failed (status word) */
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

typedef enum {
  DFLASH_ATTN_CAUSAL = 0,     /* target verification: row i sees cache slots 0..pos_i */
  DFLASH_ATTN_BLOCK_BIDIR = 1 /* draft block: every row sees the context and the whole block */
} dflash_attn_mode;

typedef enum {
  DFLASH_OP_EMBED = 0,
  DFLASH_OP_LAYER = 1,
  DFLASH_OP_FUSE = 2,
  DFLASH_OP_DRAFT = 3,
  DFLASH_OP_VERIFY = 4,
  DFLASH_OP_PATH = 5,
  DFLASH_OP_SAMPLE_DRAFTS = 6,
  DFLASH_OP_SAMPLE_ACCEPT = 7
} dflash_op;

/* Shapes and arithmetic of one decoder stack. */
typedef struct {
  int32_t hidden;       /* H */
  int32_t n_q_heads;    /* query heads */
  int32_t n_kv_heads;   /* key/value heads; n_q_heads % n_kv_heads == 0 */
  int32_t head_dim;     /* 64 or 128 */
  int32_t intermediate; /* SwiGLU width I */
  int32_t vocab;        /* V (shared embedding / LM head rows) */
  float rope_theta;     /* RoPE base (rotate-half pairing) */
  float rms_eps;        /* RMSNorm epsilon */
  int32_t dtype;        /* dflash_dtype */
} dflash_dims;

/*
 * One layer's KV cache.  Contiguous (pages == NULL): k, v each
 * [n_seqs][n_kv][capacity][head_dim].
 *
 * Paged (pages != NULL; serving-style batches whose sequences hold very
 * different lengths): k, v are page pools [pool_pages][n_kv][page_size]
 * [head_dim], and sequence s's cache slots [i*page_size, (i+1)*page_size)
 * live in pool page pages[s*max_pages + i].  capacity == max_pages *
 * page_size, page_size a multiple of 128 (one attention chunk never spans
 * two pages).  Only the pages a sequence reaches need to be mapped; a page
 * id outside [0, pool_pages) that a kernel meets raises DFLASH_ERR_INVALID_ARG
 * in the status word: its writes are skipped, its reads come from page 0.
 * With a window the ring slots (position % window) are paged the same way.
 * The arithmetic does not depend on the layout: a paged call returns what
 * the contiguous call returns, bit for bit.
 */
typedef struct {
  void* k;
  void* v;
  int32_t capacity;      /* slots per (sequence, kv head) */
  int32_t window;        /* 0: slot = position.  >0: ring of `window` slots
                            (capacity == window), slot = position % window; the
                            draft then sees the last `window` positions only. */
  const int32_t* pages;  /* NULL, or the page table [n_seqs][max_pages] */
  int32_t page_size;
  int32_t max_pages;
  int32_t pool_pages;
} dflash_kv;

typedef struct {
  const void* w_qkv;
  const void* w_o;
  const void* w_gu;
  const void* w_down;
  const void* ln1;
  const void* ln2;
} dflash_layer_weights;

/*
 * RoPE table: cos_sin[p][i] = (cos(p * w_i), sin(p * w_i)), w_i =
 * theta^(-2i/head_dim), i < head_dim/2, p < max_pos, computed on the device
 * in double and stored as float pairs ([max_pos][head_dim/2][2] floats).
 * Every call that applies RoPE reads it.
 */
int dflash_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* cos_sin,
                      dflash_stream_t stream);

/*
 * Token embedding (shared embedding, "DFlash ..." guide section 3.1: the
 * draft reuses the target's embedding and LM head).  Row i of sequence s
 * takes token first[s] for i == 0 and rest[s*(rows-1) + i-1] for i >= 1,
 * or fill_token when rest == NULL (the draft's mask tokens).
 * h[M][H] (fp32) receives the embedding rows.  A token id outside [0, V)
 * raises DFLASH_ERR_INVALID_ARG in the status word (its row reads token 0).
 */
typedef struct {
  dflash_dims dims;
  const void* embed;     /* [V][H] */
  int32_t n_seqs, rows;
  const int32_t* first;  /* [n_seqs] */
  const int32_t* rest;   /* [n_seqs][rows-1] or NULL */
  int32_t fill_token;
  float* h;              /* out [M][H] */
} dflash_embed_args;
int dflash_embed(const dflash_embed_args* a, void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * One pre-norm decoder layer, shared by the draft and the target:
 *   x = RMSNorm(h; ln1); q,k,v = x W_qkv^T; RoPE(q, k) at each row's position;
 *   o = GQA softmax attention; h += o W_o^T;
 *   x = RMSNorm(h; ln2); h += (SiLU(x W_gate^T) * (x W_up^T)) W_down^T.
 * DFLASH_ATTN_CAUSAL ("DFlash ..." guide 3.3, target verification): the
 *   rows' K/V are first written to kv at slot = position, then row i attends
 *   slots 0 .. base_pos[s] + i.  kv.window must be 0.
 * DFLASH_ATTN_BLOCK_BIDIR (guide 3.1/3.2, draft block): kv holds the
 *   injected context of positions < base_pos[s] (the last kv.window of them
 *   with a window); every row attends all of those plus every row of its own
 *   block, no mask.  The block's K/V are not stored in kv.
 * tap (optional): writes the layer's output residual, rounded to dims.dtype,
 *   to tap[row * tap_stride + tap_offset + j] (feature taps for fusion).
 * max_pos: host-side bound with base_pos[s] + rows <= max_pos for every s
 *   (sizes the attention grid; also must not exceed the RoPE table).
 * Stage outputs (each optional, NULL = not wanted; for parity checks that
 *   compare every stage with an oracle fed the GPU's own inputs): when a
 *   pointer is given the layer writes that intermediate there instead of
 *   into its workspace, so asking for it adds no work.  Every pointer must
 *   be 16-byte aligned; elements are dims.dtype.
 *     x_attn [M][H]        RMSNorm(h; ln1), the QKV projection's input
 *     q      [M][n_q*d]    rotated queries
 *     kb, vb [n_seqs][n_kv][rows][d]  the block's rotated keys and values
 *                          (DFLASH_ATTN_BLOCK_BIDIR only; causal layers
 *                          write them into kv)
 *     attn   [M][n_q*d]    attention output, the O projection's input
 *     x_mlp  [M][H]        RMSNorm(h; ln2) after the attention residual
 *     act    [M][I]        SiLU(gate) * up, the down projection's input
 */
typedef struct {
  dflash_dims dims;
  dflash_layer_weights w;
  int32_t n_seqs, rows;
  const int32_t* base_pos; /* [n_seqs] */
  float* h;                /* in/out [M][H] fp32 residual stream */
  dflash_kv kv;
  int32_t attn_mode;       /* dflash_attn_mode */
  int32_t max_pos;
  const float* rope_cs;    /* dflash_rope_table output */
  int32_t rope_max_pos;
  void* tap;               /* optional */
  int32_t tap_stride, tap_offset;
  void* out_x_attn;        /* optional stage outputs (see above) */
  void* out_q;
  void* out_kb;
  void* out_vb;
  void* out_attn;
  void* out_x_mlp;
  void* out_act;
} dflash_layer_args;
int dflash_decoder_layer_forward(const dflash_layer_args* a, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream);

/*
 * Context-feature fusion + KV injection ("DFlash ..." guide 3.2 and FAQ Q2;
 * "DFlash 2 release" news, "KV injection"): for row i < valid[s] of
 * sequence s, at position t = base_pos[s] + i, with tap features
 * f = feats[row] ([F][H], taps in increasing layer order):
 *     c_t = RMSNorm(W_fc f; fc_norm)                  (rounded to dims.dtype)
 *     for every draft layer j: K_j[t] = RoPE(W_k^j c_t, t), V_j[t] = W_v^j c_t
 * written into kv_layers[j] at slot(t).  W_k^j, W_v^j are the K and V row
 * blocks of w_qkv_layers[j].  Rows with i >= valid[s] are skipped (valid ==
 * NULL: all rows).  c_out (optional, [M][H] fp32) receives c_t.
 */
typedef struct {
  dflash_dims dims;                         /* draft dims */
  int32_t n_taps;                           /* F */
  const void* w_fc;                         /* [H][F*H] */
  const void* fc_norm;                      /* [H] */
  int32_t n_layers;                         /* <= DFLASH_MAX_LAYERS */
  const void* w_qkv_layers[DFLASH_MAX_LAYERS];
  dflash_kv kv_layers[DFLASH_MAX_LAYERS];
  const void* feats;                        /* [M][F][H] */
  int32_t n_seqs, rows;
  const int32_t* base_pos;                  /* [n_seqs] */
  const int32_t* valid;                     /* [n_seqs] or NULL */
  const float* rope_cs;
  int32_t rope_max_pos;
  float* c_out;                             /* optional */
} dflash_fuse_args;
int dflash_fuse_context(const dflash_fuse_args* a, void* ws, size_t ws_bytes,
                        dflash_stream_t stream);

/*
 * Single-step block-diffusion draft ("DFlash ..." guide 3.1): the block is
 * [anchor[s], mask, ..., mask] at positions base_pos[s] .. base_pos[s]+block-1;
 * embed -> every draft layer in DFLASH_ATTN_BLOCK_BIDIR mode over its
 * injected context -> RMSNorm(final_norm) -> shared LM head -> greedy argmax.
 * Row j >= 1 predicts the token at position base_pos[s] + j:
 * drafts[s*(block-1) + j-1] = argmax of row j (lowest index on ties).
 * With path_topk > 0 the DFlash 2 path selector (dflash_path_select) replaces
 * the drafts by its greedy path over each row's top-path_topk candidates.
 * logits (optional, [n_seqs][block-1][V] fp32) receives rows 1..block-1.
 *
 * Multi-round block denoising ("DFlash 2 release" news, "the core of DFlash
 * 2": a block diffusion model settles a block in rounds of parallel
 * denoising or correction): with denoise_rounds = R >= 2 the forward above
 * runs R times; round 1 on [anchor, mask, ...], round r >= 2 on [anchor,
 * drafts of round r-1] at the same positions, each round ending with its
 * argmax (or path walk).  drafts and logits hold the last round's.  0 and 1
 * both mean the single step; R <= DFLASH_MAX_DENOISE_ROUNDS.
 *
 * DFlash 2 two-tap dynamic depthwise convolutions (guide section 7): with
 * conv_rank = r > 0 every draft layer j carries four convolutions, at the
 * attention input (after its RMSNorm), the attention block's output (before
 * the residual add), the MLP input and the MLP output, with tap generators
 * conv_w1[j] ([4][r][H]) and conv_w2[j] ([4][2H][r]), in that order.  Over
 * the block rows u_t of a sequence: z_t = SiLU(W1 u_t), (a_t, b_t) = W2 z_t
 * (rows 0..H-1 of W2 give a, rows H..2H-1 give b), y_t = u_t + a_t u_t +
 * b_t u_{t-1} per channel with u_{-1} = 0 (block row 1 reads the anchor,
 * the last verified token).  Inputs of projections are rounded to the
 * compute type after the convolution; outputs are added to the residual.
 * r <= DFLASH_MAX_CONV_RANK.
 */
#define DFLASH_MAX_DENOISE_ROUNDS 16
#define DFLASH_MAX_CONV_RANK 128
typedef struct {
  dflash_dims dims;
  int32_t n_layers;
  dflash_layer_weights layers[DFLASH_MAX_LAYERS];
  dflash_kv kv_layers[DFLASH_MAX_LAYERS];
  const void* final_norm;                 /* [H] */
  const void* embed;                      /* [V][H] */
  const void* lm_head;                    /* [V][H] */
  int32_t n_seqs, block;
  const int32_t* anchor;                  /* [n_seqs] */
  const int32_t* base_pos;                /* [n_seqs] */
  int32_t mask_token;
  int32_t max_pos;
  const float* rope_cs;
  int32_t rope_max_pos;
  int32_t* drafts;                        /* out [n_seqs][block-1] */
  float* logits;                          /* optional */
  int32_t path_topk;                      /* 0 = off, else <= 16 */
  int32_t path_rank;                      /* R of path_u / path_v */
  const void* path_u;                     /* [R][H] */
  const void* path_v;                     /* [R][H] */
  int32_t denoise_rounds;                 /* 0 / 1 = single step, else R rounds */
  /* path selector walked by sampling (see dflash_path_select): */
  float path_temperature;                 /* 0: greedy walk */
  uint64_t path_seed;
  int32_t path_cycle;
  int32_t* path_cand_out;                 /* optional out [n_seqs][block-1][path_topk]: candidates */
  float* path_logq;                       /* optional out [n_seqs][block-1][path_topk]: log q */
  int32_t conv_rank;                      /* 0 = no convolutions */
  const void* conv_w1[DFLASH_MAX_LAYERS]; /* [4][r][H] per draft layer */
  const void* conv_w2[DFLASH_MAX_LAYERS]; /* [4][2H][r] per draft layer */
} dflash_draft_args;
int dflash_draft_block(const dflash_draft_args* a, void* ws, size_t ws_bytes,
                       dflash_stream_t stream);

/*
 * Verification + greedy acceptance ("DFlash ..." guide 3.3 and section 4
 * step 4; "DFlash 2 release" news, prefix example): from the target's last
 * residual h ([n_seqs*block][H]):
 *   g[s][i]      = argmax_v (RMSNorm(h[s,i]; final_norm) . lm_head[v])
 *   accept_len[s]= largest k <= block-1 with drafts[s][j-1] == g[s][j-1] for all j <= k
 *   out_tokens[s]= drafts[s][0..k-1], then the bonus g[s][k]
 * Ties go to the lowest vocab index; margin = top1 - top2 logit.  A NaN
 * logit raises DFLASH_ERR_NUMERIC in the status word.  drafts may be NULL
 * only when block == 1 (plain greedy decoding).
 * State update (each optional): next_anchor[s] = g[s][k];
 * commit_base[s] = base_pos[s]; commit_count[s] = k + 1;
 * base_pos[s] += k + 1.
 */
typedef struct {
  dflash_dims dims;
  const float* h;            /* [n_seqs*block][H] */
  const void* final_norm;    /* [H] */
  const void* lm_head;       /* [V][H] */
  int32_t n_seqs, block;
  const int32_t* drafts;     /* [n_seqs][block-1] */
  int32_t* argmax;           /* out [n_seqs][block] */
  float* margin;             /* out [n_seqs][block], optional */
  int32_t* accept_len;       /* out [n_seqs] */
  int32_t* out_tokens;       /* out [n_seqs][block] */
  int32_t* next_anchor;      /* optional */
  int32_t* base_pos;         /* optional in/out */
  int32_t* commit_base;      /* optional */
  int32_t* commit_count;     /* optional */
  float* logits;             /* optional [n_seqs][block][V] */
} dflash_verify_args;
int dflash_verify_accept(const dflash_verify_args* a, void* ws, size_t ws_bytes,
                         dflash_stream_t stream);

/*
 * DFlash 2 path selector, greedy walk ("DFlash ..." guide section 7): for
 * block rows j = 1..block-1 with candidate lists cand[s][j-1][0..topk-1]
 * (ranked by draft logit, best first), score(a -> b) = (U e_a) . (V e_b)
 * over the shared embedding rows e; p_0 = anchor[s]; p_j = the candidate of
 * row j with the highest score from p_{j-1} (lower rank on ties).
 * path[s][j-1] = p_j; margin (optional) = best - second-best score.
 *
 * Sampled walk (temperature > 0; the section's "greedily or by sampling"):
 * the proposal over row j's candidates is q_j(c) = softmax(score(p_{j-1},
 * c) / temperature); p_j is a Gumbel-max draw from it (Philox4x32-10 as in
 * sampling mode, purpose 5, entry = candidate rank, position base_pos[s] +
 * j); logq (optional [n_seqs][block-1][topk]) receives log q_j per
 * candidate, margin the best - second draw score.  Hand cand and logq to
 * dflash_sample_accept (draft_cand / draft_logq) for speculative sampling
 * against this proposal.
 */
typedef struct {
  dflash_dims dims;
  int32_t n_seqs, block, topk, rank;
  const void* embed;       /* [V][H] */
  const void* path_u;      /* [R][H] */
  const void* path_v;      /* [R][H] */
  const int32_t* anchor;   /* [n_seqs] */
  const int32_t* cand;     /* [n_seqs][block-1][topk] */
  int32_t* path;           /* out [n_seqs][block-1] */
  float* margin;           /* optional out [n_seqs][block-1] */
  float temperature;       /* 0: greedy walk; > 0: sampled walk */
  uint64_t seed;           /* sampled walk */
  int32_t cycle;           /* sampled walk */
  const int32_t* base_pos; /* [n_seqs] position of block row 0 (sampled walk) */
  float* logq;             /* optional out [n_seqs][block-1][topk] (sampled walk) */
} dflash_path_args;
int dflash_path_select(const dflash_path_args* a, void* ws, size_t ws_bytes,
                       dflash_stream_t stream);

/*
 * Sampling-mode verification: the lossless-in-distribution variant of the
 * greedy acceptance ("DFlash：块扩散加速的 LLM 推测解码技术", section 7: the
 * path is walked greedily or by sampling and rejection sampling keeps the
 * output distribution exactly the target's), i.e. speculative sampling at
 * temperature T > 0:
 *   q_j = softmax(draft logits of block row j / T), p_j = softmax(target
 *   logits of block row j-1 / T): both the distribution of the token at
 *   position P + j;
 *   dflash_sample_drafts draws the draft d_j of every block row j >= 1 from
 *   q_j (use the logits dflash_draft_block writes);
 *   dflash_sample_accept accepts d_j iff log u_j < log p_j(d_j) -
 *   log q_j(d_j), in order, stopping at the first rejection; it then emits a
 *   draw from max(0, p_j - q_j) normalised at that row, or -- every draft
 *   accepted -- a draw from the last target row (use the logits
 *   dflash_verify_accept writes).
 * Draws are Gumbel-max over the vocabulary.  Random numbers are Philox4x32-10
 * (Salmon et al., SC'11) with key (seed low, seed high) and counter
 * (vocabulary entry, position, sequence << 8 | purpose, cycle): give every
 * cycle its own `cycle` value.  Reductions run in a fixed order, so a call
 * is deterministic.  Token ids out of range raise DFLASH_ERR_INVALID_ARG in
 * the status word.  n_seqs * block <= 1024.
 *
 * Top-k / top-p (both calls must be given the same values): every row's
 * entries are ordered by logit (descending, lower index first on equal
 * logits); top_k > 0 keeps the first top_k, then top_p < 1 keeps the
 * shortest prefix of those whose softmax(logits / T) mass, renormalised over
 * them, reaches top_p (masses counted as floor(exp((l - max) / T) 2^32)).
 * p_j and q_j are then the renormalised softmax over each row's kept
 * entries (0 elsewhere): the output follows the filtered target
 * distribution.  top_k = 0 and top_p = 0 or 1 turn filtering off.
 */
typedef struct {
  dflash_dims dims;             /* vocab is used */
  int32_t n_seqs, block;
  float temperature;            /* > 0 */
  int32_t cycle;
  uint64_t seed;
  const int32_t* base_pos;      /* [n_seqs] position P of block row 0 */
  const float* draft_logits;    /* [n_seqs][block-1][V] */
  int32_t* drafts;              /* out [n_seqs][block-1] */
  float* draft_lse;             /* out [n_seqs][block-1]: log sum exp(logits / T) over the kept entries */
  int32_t top_k;                /* 0 = off */
  float top_p;                  /* 0 or 1 = off */
} dflash_sample_drafts_args;
int dflash_sample_drafts(const dflash_sample_drafts_args* a, void* ws, size_t ws_bytes,
                         dflash_stream_t stream);

typedef struct {
  dflash_dims dims;             /* vocab is used */
  int32_t n_seqs, block;
  float temperature;            /* > 0, as for the drafts */
  int32_t cycle;                /* as for the drafts */
  uint64_t seed;
  const float* target_logits;   /* [n_seqs][block][V] */
  const float* draft_logits;    /* [n_seqs][block-1][V] */
  const float* draft_lse;       /* [n_seqs][block-1], from dflash_sample_drafts */
  const int32_t* drafts;        /* [n_seqs][block-1] */
  int32_t* base_pos;            /* in: P; out: P + accept_len + 1 when update_base_pos */
  int32_t update_base_pos;
  int32_t* accept_len;          /* out [n_seqs] */
  int32_t* out_tokens;          /* out [n_seqs][block]: accepted drafts, the final draw, then -1 */
  int32_t* next_anchor;         /* optional out [n_seqs]: the final draw */
  int32_t* commit_base;         /* optional out [n_seqs]: P (with update_base_pos) */
  int32_t* commit_count;        /* optional out [n_seqs]: accept_len + 1 */
  int32_t top_k;                /* as for the drafts */
  float top_p;                  /* as for the drafts */
  /* Drafts from the sampled path walk: their proposal is sparse -- q_j over
   * row j's candidates, log q_j from the walk, 0 elsewhere -- and replaces
   * softmax(draft logits / T) (draft_logits / draft_lse are then unused).
   * top_k / top_p filter the target rows only. */
  int32_t draft_topk;           /* 0, or the candidates per row (<= 16) */
  const int32_t* draft_cand;    /* [n_seqs][block-1][draft_topk] */
  const float* draft_logq;      /* [n_seqs][block-1][draft_topk] */
} dflash_sample_accept_args;
int dflash_sample_accept(const dflash_sample_accept_args* a, void* ws, size_t ws_bytes,
                         dflash_stream_t stream);

/* Bytes of workspace `op` needs for these arguments (args points to the
 * op's argument struct); 0 on invalid arguments. */
size_t dflash_workspace_bytes(int32_t op, const void* args);

/* Zero a workspace (status word and the library's arrival counters). */
int dflash_workspace_init(void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Failure-detection controls kept in a workspace's header, next to its
 * status word (all zero after dflash_workspace_init, which restores the
 * defaults; dflash_read_status leaves them):
 *  - wait_limit_ns: how long a bounded device wait (a TMA copy, an MMA, a
 *    pipeline stage of another warp) spins before the kernel gives up,
 *    raises DFLASH_ERR_TIMEOUT in the status word and unwinds, keeping the
 *    GPU context usable.  0 selects the default, 1 s.
 *  - stall_kv_loads: test switches, bits: 1 makes the attention kernels issue
 *    none of their K/V copies, 2 makes the paired GEMM launch (two 256-row
 *    parts of a projection) issue none of its weight copies, so that their
 *    waits expire with nothing in flight -- the way to test the timeout path
 *    without a GPU fault.  Outputs are then meaningless.  Other bits are
 *    DFLASH_ERR_INVALID_ARG.  Keep it 0 in use.
 * The controls are copied with cudaMemcpyAsync on `stream` from host memory
 * (not inside a stream capture).  A workspace used by
 * dflash_verify_accept_noalloc has its controls reset by every such call.
 */
int dflash_workspace_control(void* ws, size_t ws_bytes, uint64_t wait_limit_ns, int32_t stall_kv_loads,
                             dflash_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's device status word.
 * *host_status receives DFLASH_OK or the first error raised on the device. */
int dflash_read_status(void* ws, dflash_stream_t stream, int32_t* host_status);

/*
 * Kernel tracing (off by default; state is per host thread).  Between
 * dflash_trace_begin and dflash_trace_pause every launch step of the library
 * (one or a few kernels of one family: a projection over several token-row
 * tiles, a GEMM and its split-K fixup) is bracketed by two CUDA events
 * recorded on its stream (event records are captured into CUDA graphs as
 * well).  dflash_trace_read, called after the traced work (or graph replay)
 * has completed, sums the event durations per kernel family into
 * stats[0 .. DFLASH_TRACE_FAMILIES-1] and returns the number of families;
 * `launches` counts the kernels launched.  `bytes` is the algorithmic DRAM traffic
 * the library attributes to the launches (weights + activations read and
 * written, each once), where it is known on the host; 0 otherwise.
 */
#define DFLASH_TRACE_FAMILIES 13
typedef struct {
  char name[24];
  int32_t launches;
  double total_ms;
  double bytes;
} dflash_trace_stat;
int dflash_trace_begin(int32_t max_launches);
int dflash_trace_pause(void);
int dflash_trace_read(dflash_trace_stat* stats, int32_t n_stats);
/* Per-step durations of the traced work in launch order: ms[i], family[i]
 * for i < min(n, count); returns count (the number of traced steps). */
int dflash_trace_launches(float* ms, int32_t* family, int32_t n);
int dflash_trace_end(void);

/*
 * Allocation-free verification + acceptance.  (No counterpart in the paper:
 * this is a deployment convenience of this library.)
 *
 * Same arguments, computation and outputs as dflash_verify_accept, but the
 * scratch memory lives in a fixed 8 MiB array inside the library's device
 * image instead of a caller-provided workspace.  It serves callers that
 * cannot allocate device memory at the point of the call: a runtime whose
 * memory is owned by a pre-sized arena or pool, a plugin that is handed
 * only input and output buffers, or code that must not allocate on its hot
 * path.  Every GPU that loads the library holds the 8 MiB array until the
 * process exits.
 *  - Runs every argument check of dflash_verify_accept first (bad arguments
 *    return DFLASH_ERR_INVALID_ARG), then rejects, with DFLASH_ERR_WORKSPACE
 *    and a message, any call whose scratch (dflash_workspace_bytes(
 *    DFLASH_OP_VERIFY, a)) exceeds 8 MiB.  That scratch is, for M =
 *    n_seqs * block token rows, G = min(SM count, ceil(V / 128) * H / 64)
 *    and BN the smallest of 16, 32, 64, 128, 256 not below min(M, 256):
 *      131328 + M*H*e + 2*G*BN*512 + G*M*12 bytes (+ up to 1 KB of
 *    alignment; e = 2 for bf16, 4 for fp32).  On a 152-SM GPU at H = 4096
 *    that admits M <= 32 token rows at any vocabulary size -- one sequence
 *    of a 16- or 17-row verification block, or two 16-row blocks -- and
 *    rejects M >= 33 (BN = 64 alone needs 9.5 MiB).
 *  - Calls no cudaMalloc/cudaFree.  The first call on a device looks up the
 *    array's device address once for that device (with it current); make
 *    that first call before any stream capture.
 *  - All calls share the one array: each call clears its status word and
 *    arrival counters first, and calls whose work overlaps on the GPU (for
 *    example on two streams at once) race.
 *  - status_out (optional, device int32) receives this call's device status
 *    bits: 0 = OK, bit 0 = a NaN reached the argmax, bit 1 = a bounded wait
 *    expired.
 */
int dflash_verify_accept_noalloc(const dflash_verify_args* a, int32_t* status_out, dflash_stream_t stream);

/* Thread-local description of the last failure. */
const char* dflash_last_error(void);

int32_t dflash_abi_version(void);

/*
 * Build variant.  The library is also built as libdflash_checked.so, with
 * device bounds assertions on the addresses its kernels compute (K/V cache
 * and query destinations of the projection epilogues, the attention's output
 * rows): a failed assertion raises DFLASH_ERR_CHECK in the status word and
 * skips the access instead of trapping.  Results are otherwise identical.
 * Independent of the variant, token ids and KV page ids read on the device
 * are always checked (DFLASH_ERR_INVALID_ARG).
 */
#define DFLASH_BUILD_CHECKED 1
int32_t dflash_build_flags(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
