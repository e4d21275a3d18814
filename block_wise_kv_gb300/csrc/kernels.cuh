// kernels.cuh — internal interface between the C ABI (dllm_api.cu) and the
// kernel translation units.  Not installed; include/dllm.h is the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dllm {

constexpr int kPage = 64;  // tokens per cache page

// Batch metadata as the kernels see it: device arrays plus the host bounds
// that every device-side check compares against.
struct BatchArgs {
  const int32_t* block_table;  // [batch][max_pages]
  const int32_t* seq_len;      // [batch]
  const int32_t* block_start;  // [batch]
  const int32_t* block_len;    // [batch]
  const int32_t* cu_block;     // [batch + 1]
  const int32_t* cu_seq;       // [batch + 1]
  int32_t* err;                // nullable error word
  int32_t batch;
  int32_t max_pages;
  int32_t num_pages;
  int32_t max_block_len;
  int32_t max_seq_len;
  int32_t total_block_rows;  // rows of x_block / q_block
  int32_t total_seq_rows;    // rows of x_full / o_full / lse
};

// Arguments of the fused projection kernel's epilogue.
struct QkvArgs {
  BatchArgs bt;
  void* k_pool;                // bf16 [P][H][64][d]
  void* v_pool;
  void* q_pool;                // boundary mode: queries of U rows
  void* q_block;               // step mode: bf16 [M][H][d]
  const float* rope;           // fp32 [rope_max_pos][d/2][2]
  int32_t rope_max_pos;
  int32_t n_heads;
  int32_t head_dim;
  int32_t d_model;
  int32_t n_tok;               // rows of x
  int32_t mode;                // kModeBlock, kModeBoundary or kModeRows
  // RMSNorm: input rows, gain, epsilon; in the workspace the normalised rows
  // x^, the per-row scale pairs and the counters of the row claims (claimed,
  // published, CTAs done)
  const void* x;               // bf16 [n_tok][d_model]
  const void* gain;            // bf16 [d_model]
  float rms_eps;
  void* xhat;                  // bf16 [n_tok][d_model]
  float2* inv;                 // [n_tok] (hi, lo) of 1 / sqrt(mean(x^2) + eps)
  int32_t* norm_ctr;           // [3]; zero before the call, zero again after it
  // stream-K schedule (n_tok <= 64): fp32 partial tiles and per-tile arrival
  // counters in the workspace; the last contributor of a tile zeroes its counter
  float* partials;             // null: one CTA per (weight tile, token tile)
  int32_t* counters;
  int32_t max_contrib;         // partial slots per weight tile
};

// Tile-packed projection weight.  Box (t, kb) = rows [128t, 128t + 128) x
// columns [64kb, 64kb + 64) of W_qkv is 16 KB contiguous at element
// ((t * boxes_per_tile + kb) * 128 + r) * 64 + c; boxes_per_tile =
// 2 * ceil(d_model / 128), columns past d_model are zero.  A CTA streaming one
// tile's K range then reads one contiguous run of memory.
inline int qkv_boxes_per_tile(int d_model) { return 2 * ((d_model + 127) / 128); }
inline size_t qkv_packed_bytes(int d_model, int n_heads, int head_dim) {
  return static_cast<size_t>(3) * n_heads * head_dim * qkv_boxes_per_tile(d_model) * 64 * 2;
}
cudaError_t launch_qkv_pack(const void* w, void* packed, int rows, int d_model, cudaStream_t stream);

// Workspace layout and schedule of the fused projection for n_tok rows:
// [counters: 4 KB][row scales: n_tok (hi, lo) pairs][x^: n_tok bf16 rows]
// [stream-K partials].  The
// counters (3 for the RMSNorm row claims, then one per output tile of a
// stream-K schedule) sit in a region of fixed size at the start, so calls of
// different shapes sharing a workspace never find another call's partials
// there; they are zero before and after every call.
constexpr size_t kQkvCounterBytes = 4096;
constexpr int kQkvNormCounters = 4;  // 3 used, the 4th keeps the tile counters 16-byte aligned
constexpr int kQkvMaxTileCounters = static_cast<int>(kQkvCounterBytes / 4) - kQkvNormCounters;
struct QkvPlan {
  int bn;            // token tile (32, 64 or 128; 256 in the wide kernel)
  bool wide;         // the persistent wide-tile kernel (qkv_wide.cu): 256 or more token rows
  bool streamk;      // stream-K over (output tile, k-unit) units, else whole tiles per CTA
  int grid;          // CTAs of the stream-K schedule / of the persistent wide kernel
  int n_tiles;       // wide kernel: output tiles (128 weight rows x 256 token rows)
  int max_contrib;   // stream-K: most CTAs sharing one output tile
  size_t inv_offset, inv_bytes, xhat_offset, xhat_bytes, part_offset, part_bytes, total_bytes;
};
QkvPlan qkv_plan(int n_tok, int d_model, int n_heads, int head_dim, int num_sms);
void qkv_wide_schedule(int n_tok, int d_model, int n_heads, int head_dim, int num_sms, QkvPlan* p);
cudaError_t launch_qkv_wide(const void* w_packed, const QkvArgs& a, const QkvPlan& plan, cudaStream_t stream);
constexpr int kModeBlock = 0;     // tokens are the packed block rows (cu_block)
constexpr int kModeBoundary = 1;  // tokens are all rows of every sequence (cu_seq)
constexpr int kModeRows = 2;      // tokens are the rows [block_start, block_start + block_len) of each
                                  // sequence (cu_block), q written to q_pool like k and v

struct AttnArgs {
  BatchArgs bt;
  const void* q_block;  // block attention: bf16 [M][H][d]
  const void* k_pool;   // bf16 [P][H][64][d]
  const void* v_pool;
  const void* q_pool;
  float* m_pool;        // fp32 [P][H][64]: written by the state build, read by the merge
  float* l_pool;
  void* o_pool;         // fp16 [P][H][64][d]: the state's O~ / l
  void* o_full;         // bf16 [R][H][d]
  float* lse;           // fp32 [R][H], nullable
  int32_t n_heads;
  int32_t head_dim;
  float scale_log2;     // softmax_scale * log2(e)
  // incremental boundary: the state of every row over the keys before its sequence's
  // current block (same layout as m_pool, l_pool, o_pool), and where the block decoded
  // last began (device int32 [batch]; the new block starts where it ended)
  float* m_pre;
  float* l_pre;
  void* o_pre;
  const int32_t* prev_start;
};

// One attention launch: a persistent grid of block-role and merge-role CTAs,
// each role walking the (sequence, head, page) units.
struct AttnPlan {
  int n_block_ctas, n_merge_ctas;  // CTAs of each role (one CTA per SM in all)
  size_t total_bytes;              // workspace (none needed: 0)
};
AttnPlan attn_plan(int batch, int n_heads, int head_dim, int max_seq_len, int max_block_len, int total_seq_rows,
                   int total_block_rows, int num_sms, bool block, bool merge);
bool attn_batch_supported(int batch);

// ---- launchers (return the first CUDA error, cudaSuccess otherwise) ------
// Each launcher encodes the TMA tensor maps it needs from the raw pointers.
cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, double theta, cudaStream_t stream);
cudaError_t launch_zero_tails(const BatchArgs& bt, void* k_pool, void* v_pool, void* q_pool, int n_heads,
                              int head_dim, cudaStream_t stream);
cudaError_t launch_qkv_gemm(const void* w_packed, const QkvArgs& a, const QkvPlan& plan, cudaStream_t stream);
// The block attention (LaCache Eq. (2)-(6) over all keys of each block row)
// and/or the FACache merge of every invariant row, as planned by attn_plan.
cudaError_t launch_step_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);
// The block-only epilogue (lm_head.cu): the block rows of the final hidden states, the
// final RMSNorm, the LM head and the softmax over the vocabulary.
struct LmArgs {
  BatchArgs bt;
  const void* h;     // bf16 [R][d_model]: every row's final hidden state (packed by cu_seq)
  const void* gain;  // bf16 [d_model]: the final RMSNorm gain
  void* xhat;        // workspace: bf16 [n_rows][d_model]
  float* pmax;       // workspace: [2 * vocab tiles][n_rows] per-half-tile max, sum of exp, argmax
  float* psum;
  int32_t* parg;
  void* logits;      // bf16 [n_rows][vocab], nullable
  float* lse;        // [n_rows]
  int32_t* argmax;   // [n_rows]
  float* p_max;      // [n_rows]
  int32_t n_rows, d_model, vocab;
  float rms_eps;
};
size_t lm_head_workspace_bytes(int n_rows, int d_model, int vocab);
void lm_bind_workspace(LmArgs* a, void* ws);
cudaError_t launch_lm_head(const void* w_lm, const LmArgs& a, int num_sms, cudaStream_t stream);

// The rest of the layer for the block rows (ffn.cu): output projection + residual, AddNorm
// with per-group e4m3 quantisation, the FP8 gate-up GEMM with SwiGLU and requantisation, the
// FP8 down GEMM + residual.
struct FfnArgs {
  BatchArgs bt;
  const void* o_full;   // bf16 [R][H d]: the attention output of every row
  const void* x_block;  // bf16 [M][d_model]: the layer input of the block rows (first residual)
  const void* gain2;    // bf16 [d_model]: the FFN's RMSNorm gain
  void* y;              // bf16 [M][d_model]: the layer output of the block rows
  void* o_block;        // workspace: bf16 [M][H d]
  void* h1;             // workspace: bf16 [M][d_model]
  void* x2;             // workspace: e4m3 [M][d_model]
  float* x2_scale;      // workspace: [M][d_model / 128]
  int32_t n_rows, d_model, hd, d_ff;
  float rms_eps;
};
struct FfnWeights {
  const void* w_o;         // bf16 [d_model][H d]
  const void* w_gu;        // e4m3 [2 d_ff][d_model]: row 2j gate j, row 2j + 1 up j
  const float* gu_scale;   // [2 d_ff / 128][d_model / 128]
  const void* w_down;      // e4m3 [d_model][d_ff]
  const float* down_scale; // [d_model / 128][d_ff / 128]
};
// One token-major GEMM of ffn.cu.
struct DenseArgs {
  int32_t M, N, K, splits;
  const float* sa;   // e4m3 A: [M][K / 128] row group scales
  const float* sb;   // e4m3 B: [N / 128][K / 128] block scales
  float* part;       // [splits][M][N] fp32 partial sums
  void* out8;        // SwiGLU: e4m3 [M][N / 2]
  float* out_scale;  // SwiGLU: [M][N / 2 / 128]
  int32_t* err;
};
size_t ffn_workspace_bytes(int n_rows, int d_model, int hd, int d_ff, int num_sms);
cudaError_t launch_ffn(const FfnArgs& a, const FfnWeights& w, void* ws, int num_sms, cudaStream_t stream);

// Attention of 128-row query tiles on the tensor cores (attn_rows.cu):
//   kRowsState  every row of U over the keys of U: (m, l, O~) into the pools (the cache build)
//   kRowsBlock  the block rows over every key: O and L (blocks of more than 64 rows)
//   kRowsMerge  every row of U over the block keys, merged with its cached state: O and L
//   kRowsStatePre  as kRowsState, and the state over the keys before the block into the pre pools
//   kRowsAdvOld    incremental boundary, rows kept from the last one: pre extended by the decoded
//                  block's keys, then the state over U from it and the suffix keys
//   kRowsAdvNew    incremental boundary, the decoded rows: pre over the keys before the new
//                  block, then the state over U from it and the suffix keys
constexpr int kRowsState = 0;
constexpr int kRowsBlock = 1;
constexpr int kRowsMerge = 2;
constexpr int kRowsStatePre = 3;
constexpr int kRowsAdvOld = 4;
constexpr int kRowsAdvNew = 5;
cudaError_t launch_rows_attention(const AttnArgs& a, int mode, int num_sms, cudaStream_t stream);

}  // namespace dllm
