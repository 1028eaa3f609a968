// internal.h -- launch interface between the C-ABI layer (abi.cu) and the
// kernel translation units.  Host-side declarations only.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dfl {

enum EpiKind : int32_t {
  EPI_STORE = 0,   // out_f32[m][n] = acc
  EPI_RESID = 1,   // out_f32[m][n] += acc
  EPI_QKV = 2,     // rows = [Q heads | K heads | V heads]: RoPE, then q_out / KV destinations
  EPI_SWIGLU = 3,  // rows = [gate | up]: act[m][j] = SiLU(gate_j) * up_j
};

constexpr int kMaxSeg = 16;

// One GEMM problem Y[m][n] = sum_k X[m][k] W[n][k] with a fused epilogue.
// Several weight segments may share one launch (K/V injection into every
// draft layer); segment s covers output rows [0, seg_rows) of weight
// seg_w[s] starting at row seg_row0.
struct GemmDesc {
  int dtype;                  // DFLASH_F32 / DFLASH_BF16 (X, W, outputs)
  int M, K;                   // token rows, reduction length
  const void* X;              // [M][K]
  int nseg;
  const void* seg_w[kMaxSeg]; // weight base pointers ([rows][K])
  int seg_row0;               // first weight row used in every segment
  int seg_rows;               // output rows per segment
  int kind;                   // EpiKind
  // row map
  const int32_t* base_pos;
  const int32_t* valid;
  int rows;                   // rows per sequence
  // EPI_STORE / EPI_RESID
  float* out_f32;
  int ldo;
  // EPI_QKV
  void* q_out;                // [M][nq*d] or null when seg_row0 skips Q
  int nq, nkv, d;
  void* k_dst[kMaxSeg];
  void* v_dst[kMaxSeg];
  int kv_cap, kv_window;
  int kv_slot_mode;           // 0: slot = in-block row index (block scratch); 1: slot = position (cache)
  const float* rope_cs;
  int rope_max_pos;
  // EPI_SWIGLU
  void* act_out;              // [M][inter]
  int inter;
};

// DFlash 2 dynamic depthwise convolution over M token rows (rows per
// sequence = `rows`): z = SiLU(W1 u) into z [M][r], then y = u + a u + b u_prev
// with (a, b) = W2 z; out = round(y) (resid = 0, out of the compute type) or
// out += y (resid = 1, out and u fp32).
struct ConvDesc {
  int dtype;
  int M, H, r, rows;
  const void* w1;   // [r][H]
  const void* w2;   // [2H][r]
  const void* u;    // [M][H]: compute type (resid = 0) or fp32 (resid = 1)
  void* out;        // [M][H]
  int resid;
  float* z;         // [M][r] scratch
};
cudaError_t launch_dyn_conv(const ConvDesc& c, cudaStream_t st);

// Paged KV caches: copy the K/V rows that a projection wrote into the
// contiguous block scratch [S][nkv][rows][d] (per layer) to their cache
// slots in the page pools.  Row m of sequence s = m / rows is copied when it
// is live (valid), its position base_pos[s] + m % rows lies in
// [0, rope_max_pos) and its slot (position, or position % window) is below
// the capacity -- the rows the projection's epilogue wrote.
struct KvScatter {
  int dtype, n_layers, S, rows, nkv, d;
  const int32_t* base_pos;
  const int32_t* valid;
  int window, cap, rope_max_pos;
  const void* kb[kMaxSeg];
  const void* vb[kMaxSeg];
  void* kpool[kMaxSeg];
  void* vpool[kMaxSeg];
  const int32_t* pages[kMaxSeg];
  int ps, max_pages, pool;
  uint32_t* status;
};
cudaError_t launch_kv_page_scatter(const KvScatter& k, cudaStream_t st);

// Attention problem (see dflash_decoder_layer_forward).
struct AttnDesc {
  int dtype;
  int mode;                   // dflash_attn_mode
  int n_seqs, rows, nq, nkv, d;
  const int32_t* base_pos;
  const void* q;              // [M][nq*d]
  const void* kc;             // cache [S][nkv][cap][d], or a page pool [pool][nkv][ps][d]
  const void* vc;
  int cap, window;
  const int32_t* pages;       // page table [S][max_pages] (paged caches) or null
  int ps, max_pages, pool;
  const void* kb;             // block scratch [S][nkv][rows][d] (bidir)
  const void* vb;
  void* out;                  // [M][nq*d]
  int max_pos;                // bound on base_pos + rows
  float* partials;            // workspace
  uint32_t* counters;
  uint32_t* status;
};

struct HeadDesc {
  int dtype;
  int M, H, V;
  const void* x;              // [M][H] normalised, rounded
  const void* w;              // [V][H]
  int n_seqs, block;
  int mode;                   // 0: draft (argmax rows 1..block-1 -> drafts), 1: verify, 2: draft top-k
  int topk;
  const int32_t* drafts;      // verify
  int32_t* drafts_out;        // draft
  int32_t* argmax;            // verify
  float* margin;
  int32_t* accept_len;
  int32_t* out_tokens;
  int32_t* next_anchor;
  int32_t* base_pos;
  int32_t* commit_base;
  int32_t* commit_count;
  int32_t* cand_out;          // top-k mode [S][block-1][topk]
  float* logits;              // optional [M][V] (draft: rows 1.. only written)
  float* partials;            // workspace
  uint32_t* counters;
  uint32_t* status;
};

struct PathDesc {
  int dtype;
  int n_seqs, block, topk, rank, H, V;
  const void* embed;
  const void* u;
  const void* v;
  const int32_t* anchor;
  const int32_t* cand;        // [S][block-1][topk]
  int32_t* path;
  float* margin;
  float* proj;                // workspace [S][1 + (block-1)*topk][2*rank]: U e, V e per token slot
  uint32_t* status;
  // sampled walk (T > 0): Philox draws, the proposal's log-probabilities
  float T;                    // 0: greedy walk
  uint64_t seed;
  int cycle;
  const int32_t* base_pos;    // [S] position of block row 0
  float* logq;                // optional out [S][block-1][topk]
  int32_t* cand_out;          // optional out [S][block-1][topk]: the candidate lists walked
};

// Sampling-mode verification (k_sample.cu).
// Kept set of one logit row under top-k / top-p: the entries up to (key,
// idx) in the order (logit descending, index ascending); see k_sample.cu.
struct RowFilter {
  uint32_t key;
  int idx;
};

struct SampleDesc {
  int n_seqs, block, V, cycle;
  float T;
  int top_k;                  // 0 = off
  float top_p;                // 1 = off
  const RowFilter* filt_t;    // [S][block] target rows' kept sets (filtering), else null
  const RowFilter* filt_d;    // [S][block-1] draft rows' kept sets (acceptance, filtering), else null
  RowFilter* filt_d_out;      // [S][block-1] (draft draws, filtering)
  int qk;                     // sparse proposal (the sampled path walk): candidates per row, else 0
  const int32_t* qcand;       // [S][block-1][qk]
  const float* qlogq;         // [S][block-1][qk] log q over the candidates
  uint64_t seed;
  int32_t* base_pos;          // [S] position of block row 0 (advanced when update_base)
  const float* draft_logits;  // [S][block-1][V]
  const float* target_logits; // [S][block][V]
  const float* draft_lse;     // [S][block-1] (acceptance)
  float* draft_lse_out;       // [S][block-1] (draft draws)
  int32_t* drafts_out;        // [S][block-1] (draft draws)
  const int32_t* drafts;      // [S][block-1] (acceptance)
  int32_t* out_tokens;
  int32_t* accept_len;
  int32_t* next_anchor;
  int32_t* commit_base;
  int32_t* commit_count;
  int update_base;
  int32_t* seq_k;             // workspace [S]
  void* part;                 // workspace, sample_part_bytes(rows)
  uint32_t* counters;
  uint32_t* status;
};
size_t sample_part_bytes(int rows);
cudaError_t launch_sample_drafts(const SampleDesc& d, cudaStream_t st);
cudaError_t launch_sample_accept(const SampleDesc& d, float* lse_t, cudaStream_t st);

// Path-selector projection scratch (floats) for S sequences.
inline size_t path_proj_floats(int S, int block, int topk, int rank) {
  return (size_t)S * (1 + (size_t)(block - 1) * topk) * 2 * rank;
}

// elementwise
cudaError_t launch_rope_table(float theta, int d, int max_pos, float* cs, cudaStream_t st);
cudaError_t launch_embed(int dtype, const void* E, int H, int V, int n_seqs, int rows, const int32_t* first,
                         const int32_t* rest, int fill, float* h, uint32_t* status, cudaStream_t st);
cudaError_t launch_rmsnorm(int dtype, const float* h, const void* g, int M, int H, float eps,
                           void* x_out, cudaStream_t st);
cudaError_t launch_to_f32(int dtype, const void* src, size_t n, float* dst, cudaStream_t st);
cudaError_t launch_store_tap(int dtype, const float* h, int M, int H, void* tap, int stride,
                             int offset, cudaStream_t st);

// GEMM (SIMT path; fp32 and bf16)
cudaError_t launch_gemm_simt(const GemmDesc& g, cudaStream_t st);
int gemm_out_rows(const GemmDesc& g);

// GEMM (tcgen05 path; bf16).  ws/ws_bytes: split-K partials; counters.
size_t gemm_tc_workspace(const GemmDesc& g, int num_sms);
cudaError_t launch_gemm_tc(const GemmDesc& g, void* ws, size_t ws_bytes, uint32_t* counters,
                           uint32_t* status, int num_sms, cudaStream_t st);
bool gemm_tc_supported(const GemmDesc& g);

// attention
size_t attn_workspace(const AttnDesc& a);
cudaError_t launch_attention(const AttnDesc& a, cudaStream_t st);

// LM head + argmax / accept / top-k
size_t head_workspace(const HeadDesc& h, int num_sms);
cudaError_t launch_head(const HeadDesc& h, int num_sms, cudaStream_t st);
cudaError_t launch_head_simt(const HeadDesc& h, int num_sms, cudaStream_t st);
bool head_tc_supported(const HeadDesc& h);
size_t head_tc_workspace(const HeadDesc& h, int num_sms);
cudaError_t launch_head_tc(const HeadDesc& h, int num_sms, cudaStream_t st);

// path selector
cudaError_t launch_path_select(const PathDesc& p, cudaStream_t st);
// Top-k mode of the draft head: the per-tile lists of the tensor-core head
// (tlist, n_tiles), or the logit rows h.logits of the CUDA-core head (tlist
// NULL), merged into h.cand_out [S][block-1][topk].
cudaError_t launch_topk_merge(const HeadDesc& h, const void* tlist, int n_tiles, cudaStream_t st);
// The tensor-core head's per-tile top-k lists inside h.partials.
const void* head_tc_tlist(const HeadDesc& h, int num_sms, int* n_tiles);

}  // namespace dfl
