/* dllm.h — C ABI of the GB300 (sm_103a) per-layer inner denoising step of
 * block-wise (semi-autoregressive) diffusion-LLM decoding.
 *
 * One inner step of one layer, for a batch of sequences that are each in the
 * middle of decoding block C_b = [s_b, s_b + B_b) of N_b tokens:
 *
 *   dllm_block_qkv_rope_write  RMSNorm -> QKV projection -> RoPE for the B_b
 *                              block rows only, with K/V written once into the
 *                              paged bf16 cache and Q into q_block.
 *   dllm_block_attention       bidirectional attention of the block rows over
 *                              [prefix KV | fresh block KV | suffix KV].
 *   dllm_state_merge           output rows of the invariant set U (prefix and
 *                              suffix): cached online-softmax state (m, l, O~)
 *                              merged exactly with the fresh block keys.
 *   dllm_step_attention        both of the previous two in one launch.
 *
 * and, once per block boundary, dllm_cache_build, which fills the paged cache
 * for all rows and the per-row state (m, l, O~) of every row of U over the
 * keys of U.  Sources (page titles):
 *   - "LaCache: Exact Caching and Precision-Adaptive Inference for Diffusion
 *     Large Language Models": §3.3.2 Eq. (1) (token-wise operators and their
 *     cache), §3.3.3 Eq. (2)-(6) and Algorithm 1 (FACache).
 *   - "Flash-dLLM: IO-aware KV caching ..." news write-up, section
 *     "Flash-Cache: Fusing Projection, RoPE, and Cache Writes into One Kernel"
 *     (fused projection + RoPE + single KV write; block table for ragged
 *     batches; flat pre-allocated cache).
 *   - "Fast-dLLM Block-wise DualCache" docs: sections "Block-wise Generation",
 *     "DualCache Data Structure", "Building the Dual Cache Manually".
 *
 * Conventions for every entry point
 *   - Memory: the caller owns every buffer.  The library allocates nothing and
 *     keeps no global mutable state.  Pointers named "device" must be device
 *     memory of the current device; structs are read on the host during the
 *     call only.
 *   - Execution: asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream).  No call synchronises or reads device
 *     memory on the host; host scalars in dllm_batch size the launch grids.
 *   - Errors: arguments are validated on the host before any launch; on a
 *     failed validation the call returns a non-zero status and launches
 *     nothing.  A launch failure returns DLLM_ERR_CUDA.  Device-side checks
 *     (block-table entries outside [0, num_pages), per-sequence metadata that
 *     contradicts the host bounds, a bounded wait that ran out, a cached state
 *     beyond its storage range) skip the offending access and OR a
 *     DLLM_DEVERR_* bit into *batch->error_flag
 *     when that pointer is non-NULL; outputs are then undefined.
 *   - Thread safety: calls on different streams are safe when their outputs
 *     do not overlap.
 *   - Overlap with the preceding kernel: the calls are launched with
 *     programmatic dependent launch.  The attention calls
 *     (dllm_block_attention, dllm_state_merge, dllm_step_attention) may read
 *     the batch metadata, the block table, q_pool, m_pool, l_pool, o_pool and
 *     every k/v page that holds none of the current blocks' rows before the
 *     kernel that precedes them on the stream has finished; that kernel must
 *     not write those.  dllm_block_qkv_rope_write writes only q_block and the
 *     current blocks' k/v rows, so the step's own order (projection, then
 *     attention) meets this.  q_block and the current blocks' k/v pages are
 *     read only after the preceding kernel has completed.  The projection
 *     calls (dllm_cache_build, dllm_block_qkv_rope_write) may read w_packed
 *     and rms_gain before the preceding kernel has finished; that kernel
 *     must not write them.  Everything else they read or write is touched
 *     only after the preceding kernel has completed.
 *
 * Layouts (all row-major, little-endian, bf16 = IEEE bfloat16)
 *   page      = 64 consecutive token positions of one sequence.
 *   k_pool, v_pool, q_pool: bf16 [num_pages][n_heads][64][head_dim]
 *   m_pool, l_pool:         fp32 [num_pages][n_heads][64]
 *   o_pool:                 fp16 [num_pages][n_heads][64][head_dim] (the state's O~ / l)
 *   token at position p of sequence b lives at page block_table[b][p / 64],
 *   slot p % 64.
 *   w_qkv:   bf16 [3 * n_heads * head_dim][d_model]; rows are Q heads, then K
 *            heads, then V heads, head-major, head_dim rows per head.  The
 *            projection calls read it in the tile-packed form w_packed
 *            written once per layer by dllm_qkv_weight_pack:
 *   w_packed: bf16; box (t, kb) = rows [128t, 128t+128) x columns
 *            [64kb, 64kb+64) of w_qkv is stored contiguously (row-major
 *            128 x 64) at element ((t * KB + kb) * 128) * 64, with
 *            KB = 2 * ceil(d_model / 128) boxes per 128-row tile and zeros in
 *            the columns past d_model.
 *   rms_gain: bf16 [d_model].
 *   rope_table: fp32 [rope_max_pos][head_dim / 2][2] = (cos, sin) of
 *            p * rope_theta^(-2i/head_dim); filled by dllm_rope_table_build.
 *   x_block, q_block: rows of the current blocks packed in sequence order,
 *            cu_block[b] .. cu_block[b+1]-1.  x_block bf16 [M][d_model],
 *            q_block bf16 [M][n_heads][head_dim].
 *   x_full, o_full: all rows of all sequences packed in sequence order,
 *            cu_seq[b] .. cu_seq[b+1]-1.  x_full bf16 [R][d_model],
 *            o_full bf16 [R][n_heads][head_dim], lse fp32 [R][n_heads].
 */
#ifndef DLLM_H_
#define DLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dllm_status {
  DLLM_OK = 0,
  DLLM_ERR_INVALID_ARGUMENT = 1,     /* NULL/misaligned pointer, inconsistent sizes */
  DLLM_ERR_UNSUPPORTED = 2,          /* head_dim not in {64,128}, page_size != 64, ... */
  DLLM_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below dllm_workspace_size() */
  DLLM_ERR_CUDA = 4,                 /* a CUDA runtime/driver call or launch failed */
  DLLM_ERR_TIMEOUT = 5               /* reserved for host-observed device timeouts */
} dllm_status;

/* Bits a kernel ORs into *dllm_batch.error_flag (device int32). */
#define DLLM_DEVERR_TIMEOUT 1   /* a bounded on-chip wait gave up */
#define DLLM_DEVERR_BAD_PAGE 2  /* block_table entry outside [0, num_pages) */
#define DLLM_DEVERR_BAD_SHAPE 4 /* seq_len/block_start/block_len/cu_* contradict the host bounds */
#define DLLM_DEVERR_RANGE 8     /* a state's O~ / l beyond fp16 range (a value above 65504 in magnitude) */

/* Shape of one attention layer. */
typedef struct dllm_layer_desc {
  int32_t d_model;     /* D: multiple of 64 */
  int32_t n_heads;     /* H: H*head_dim must be a multiple of 128 */
  int32_t head_dim;    /* d: 64 or 128 */
  int32_t page_size;   /* tokens per cache page: must be 64 */
  float rope_theta;    /* RoPE base (e.g. 10000, 500000) */
  float rms_eps;       /* RMSNorm epsilon */
  float softmax_scale; /* scale of q.k; 0 selects 1/sqrt(head_dim) */
} dllm_layer_desc;

/* The paged cache of one layer (device buffers, caller-owned). */
typedef struct dllm_cache {
  void* k_pool;      /* bf16 [num_pages][H][64][d]: RoPE'd keys of every position */
  void* v_pool;      /* bf16 [num_pages][H][64][d]: values */
  void* q_pool;      /* bf16 [num_pages][H][64][d]: RoPE'd queries of U rows */
  float* m_pool;     /* fp32 [num_pages][H][64]: cached row max over U keys (natural units of scale*q.k) */
  float* l_pool;     /* fp32 [num_pages][H][64]: cached sum of exp(S - m) over U keys */
  void* o_pool;      /* fp16 [num_pages][H][64][d]: cached O~ / l, O~ = sum of exp(S - m) v over U keys
                      * (the state is kept normalised: O~ = l * o_pool) */
  int32_t num_pages; /* pages in each pool; num_pages*H*64 < 2^31 */
  /* Optional (all NULL, or all set): the prefix state of each row, the same
   * (m, l, O~ / l) over only the keys before its sequence's current block, in
   * the layouts and types of m_pool, l_pool, o_pool.  dllm_cache_build fills it when set;
   * dllm_cache_advance needs it. */
  float* m_pre;
  float* l_pre;
  void* o_pre;
} dllm_cache;

/* A ragged batch.  Host scalars bound the device arrays and size the grids. */
typedef struct dllm_batch {
  int32_t batch;             /* number of sequences (>= 0) */
  int32_t max_pages_per_seq; /* row stride of block_table; >= ceil(N_b / 64) for every b */
  int32_t total_block_rows;  /* M = sum_b B_b = cu_block[batch] */
  int32_t total_seq_rows;    /* R = sum_b N_b = cu_seq[batch] */
  int32_t max_block_len;     /* >= every B_b; at most 64 */
  int32_t max_seq_len;       /* >= every N_b */
  const int32_t* block_table; /* device int32 [batch][max_pages_per_seq]: physical page ids */
  const int32_t* seq_len;     /* device int32 [batch]: N_b >= 1 */
  const int32_t* block_start; /* device int32 [batch]: s_b, 0 <= s_b, s_b + B_b <= N_b */
  const int32_t* block_len;   /* device int32 [batch]: B_b, 1 <= B_b <= max_block_len */
  const int32_t* cu_block;    /* device int32 [batch + 1]: prefix sums of B_b */
  const int32_t* cu_seq;      /* device int32 [batch + 1]: prefix sums of N_b */
  int32_t* error_flag;        /* device int32, nullable: DLLM_DEVERR_* bits are ORed in */
} dllm_batch;

/* Operation ids for dllm_workspace_size. */
#define DLLM_OP_CACHE_BUILD 0
#define DLLM_OP_BLOCK_QKV_ROPE_WRITE 1
#define DLLM_OP_BLOCK_ATTENTION 2
#define DLLM_OP_STATE_MERGE 3
#define DLLM_OP_STEP_ATTENTION 4
#define DLLM_OP_CACHE_ADVANCE 5 /* pass the decoded blocks' dllm_batch */

/* Bytes of device workspace `op` needs for this layer and batch (0 if none).
 * The workspace is scratch owned by the caller, 256-byte aligned, and may be
 * reused once the call's work on its stream has completed. */
dllm_status dllm_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t op, size_t* bytes);

/* Fill the RoPE table (device fp32 [max_pos][head_dim/2][2]) with
 * (cos, sin) of p * rope_theta^(-2i/head_dim), computed in fp64 on the device
 * and rounded to fp32.  RoPE: LaCache Eq. (1); rotate-half pairs (i, i+d/2). */
dllm_status dllm_rope_table_build(const dllm_layer_desc* desc, int32_t max_pos, float* rope_table, void* stream);

/* Bytes of the tile-packed projection weight of this layer shape:
 * 3 * n_heads * head_dim * 2 * ceil(d_model / 128) * 64 * 2. */
dllm_status dllm_qkv_weight_packed_bytes(const dllm_layer_desc* desc, size_t* bytes);

/* Write the tile-packed copy of w_qkv (layout above) that dllm_cache_build and
 * dllm_block_qkv_rope_write read.  A pure reordering (bit-exact), done once
 * per layer when the weights are loaded, so that every projection streams
 * whole 16 KB runs of weight memory (no counterpart in the pages: a layout
 * choice of this library).  w_qkv and w_packed: device, 16-byte aligned,
 * not overlapping; w_packed holds dllm_qkv_weight_packed_bytes bytes. */
dllm_status dllm_qkv_weight_pack(const dllm_layer_desc* desc, const void* w_qkv, void* w_packed, void* stream);

/* Block boundary (LaCache Algorithm 1 with GenStep = True; Fast-dLLM
 * compute_block_dual_cache).  For every row of every sequence:
 *   x^ = RMSNorm(x) (correctly rounded to bf16), [q k v] = x^ W_qkv^T (fp32
 *   accumulation), RoPE(q, k) at position p, and k, v (and q for rows of U)
 *   written as bf16 into the pools.  Pool positions p >= N_b of each
 *   sequence's last page are set to zero.
 * Then for every row r of U_b = [0, N_b) \ [s_b, s_b + B_b) and head h, the
 * online-softmax state over the keys of U_b only (LaCache §3.3.3):
 *   m = max_{j in U} S_rj, l = sum_{j in U} exp(S_rj - m),
 *   O~ = sum_{j in U} exp(S_rj - m) v_j,   S_rj = scale * q_r . k_j,
 * written to m_pool, l_pool and (as O~ / l, rounded to fp16) o_pool at row r's
 * slot.  If U_b is empty for a row's keys, m = -inf, l = 0, o_pool = 0.  When the cache's prefix state pools
 * are set, the same state over only the keys [0, s_b) is written there too
 * (what dllm_cache_advance extends).
 *   x_full: device bf16 [R][d_model]; rms_gain: device bf16 [d_model];
 *   w_packed: device, from dllm_qkv_weight_pack; rope_table: device fp32, rope_max_pos
 *   >= max_seq_len positions; ws: device scratch of
 *   dllm_workspace_size(DLLM_OP_CACHE_BUILD) bytes. */
dllm_status dllm_cache_build(const dllm_layer_desc* desc, const dllm_batch* batch, const void* x_full,
                             const void* rms_gain, const void* w_packed, const float* rope_table, int32_t rope_max_pos,
                             const dllm_cache* cache, void* ws, size_t ws_bytes, void* stream);

/* Incremental block boundary: the cache of dllm_cache_build for the next
 * blocks, when only the just-decoded blocks' rows changed since the last
 * boundary (the state of every other row is rebuilt from cached pieces, per
 * KV block: LaCache §3.3.3, the exact merge of partial states; Fast-dLLM
 * "Block-wise Generation": blocks are decoded left to right, each new block
 * starting where the decoded one ended).
 *   batch:   the new blocks (block_start s_b', block_len B_b').
 *   decoded: the blocks just decoded: the same sequences, block_table,
 *            seq_len and cu_seq pointers and host bounds as batch, with
 *            block_start s_b, block_len = s_b' - s_b, cu_block over those
 *            lengths (0 <= s_b < s_b').
 *   x_decoded: device bf16 [decoded->total_block_rows][d_model], the final
 *            rows of the decoded blocks, packed like x_block.
 *   cache:   written by dllm_cache_build (with the prefix state pools set)
 *            and any number of dllm_cache_advance calls since; every row
 *            outside the decoded blocks must be the one the cache was built
 *            from.
 * In order: the decoded rows' q, k, v (RMSNorm, projection, RoPE) into the
 * pools; for every row r of U' = [0, s_b') u [s_b' + B_b', N_b):
 *   pre'(r)   = pre(r) merged with r's partial state over the decoded keys
 *               [s_b, s_b') (rows kept from the last boundary), or r's state
 *               over [0, s_b') (the decoded rows);
 *   state'(r) = pre'(r) merged with r's partial state over [s_b' + B_b', N_b)
 * written to m_pre/l_pre/o_pre and m_pool/l_pool/o_pool.  The result equals
 * dllm_cache_build on the same rows up to the rounding order of the sums and
 * the fp16 rounding of the stored O~ / l that the kept rows extend.
 *   ws: dllm_workspace_size(desc, decoded, DLLM_OP_CACHE_ADVANCE) bytes. */
dllm_status dllm_cache_advance(const dllm_layer_desc* desc, const dllm_batch* batch, const dllm_batch* decoded,
                               const void* x_decoded, const void* rms_gain, const void* w_packed,
                               const float* rope_table, int32_t rope_max_pos, const dllm_cache* cache, void* ws,
                               size_t ws_bytes, void* stream);

/* Inner step, part 1 (LaCache §3.3.2 Eq. (1); Flash-dLLM Flash-Cache): for
 * the B_b rows of each current block only, in one kernel: x^ = RMSNorm(x_block)
 * correctly rounded to bf16, [q k v] = x^ W_qkv^T with fp32 accumulation,
 * RoPE(q, k) at absolute position p = s_b + i, then one write: k, v as bf16
 * into k_pool / v_pool at (block_table[b][p/64], h, p%64) and q as bf16 into
 * q_block [M][H][d].
 *   x_block: device bf16 [M][d_model]; q_block: device bf16 [M][H][d];
 *   w_packed: device, from dllm_qkv_weight_pack;
 *   ws: dllm_workspace_size(DLLM_OP_BLOCK_QKV_ROPE_WRITE) bytes, 256-byte
 *   aligned: 1 KB of counters, one fp32 pair per row (the RMSNorm scale
 *   1 / sqrt(mean(x^2) + eps) as hi + lo), the bf16 x^ rows [M][d_model]
 *   (each region 256-byte aligned), then, for small models, the fp32 partial
 *   tiles of a split schedule.  The counters must be zero before the
 *   workspace's first use; every call leaves them zero (also after a
 *   device-side timeout).  The same holds for dllm_cache_build's workspace
 *   (with R rows). */
dllm_status dllm_block_qkv_rope_write(const dllm_layer_desc* desc, const dllm_batch* batch, const void* x_block,
                                      const void* rms_gain, const void* w_packed, const float* rope_table,
                                      int32_t rope_max_pos, const dllm_cache* cache, void* q_block, void* ws,
                                      size_t ws_bytes, void* stream);

/* The same call as dllm_block_qkv_rope_write for callers that cannot
 * allocate device memory (no counterpart in the pages; an addition of this
 * library).  Some callers cannot hand the library a workspace: a plugin host
 * that passes only inputs and outputs, a server with a fixed memory budget
 * reserved at start-up that forbids allocation on the serving path, or code
 * running where cudaMalloc is not allowed.  This variant allocates nothing and
 * takes no workspace: its scratch is a fixed 8 MiB array in the library's own
 * device memory (held by every GPU that loads the library until exit), so the
 * call's dllm_workspace_size(DLLM_OP_BLOCK_QKV_ROPE_WRITE) must not exceed
 * 8 MiB (about 0.26 MiB for 32 block rows of d_model 4096: mostly the x^
 * rows); a larger need returns DLLM_ERR_WORKSPACE_TOO_SMALL and launches
 * nothing.  The first call
 * on each device looks up the array's device address with that device
 * current (make that first call before any stream capture) and keeps it for the
 * life of the process: after cudaDeviceReset on a device the array may move,
 * so do not call this entry point on a device again after resetting it.  All
 * calls share
 * the array: calls whose GPU work may overlap (different streams without
 * ordering) race on it.  Arguments, layouts and results are otherwise those
 * of dllm_block_qkv_rope_write. */
dllm_status dllm_block_qkv_rope_write_noalloc(const dllm_layer_desc* desc, const dllm_batch* batch,
                                              const void* x_block, const void* rms_gain, const void* w_packed,
                                              const float* rope_table, int32_t rope_max_pos,
                                              const dllm_cache* cache, void* q_block, void* stream);

/* Inner step, part 2 (LaCache Eq. (2)-(6); Fast-dLLM DualCache "Inner step on
 * block k"): for each block row i of sequence b and head h,
 *   O = sum_j softmax_j(scale * q_i . k_j) v_j over ALL keys j in [0, N_b)
 * read through block_table (prefix | fresh block | suffix), written as bf16 to
 * o_full row cu_seq[b] + s_b + i, and L = m + ln l to lse (nullable) at the
 * same row.  q_block as written by dllm_block_qkv_rope_write; the pools as
 * written by dllm_cache_build and this step's dllm_block_qkv_rope_write.
 * The online-softmax state of a row runs over all pages of its sequence
 * (Eq. (2)-(6)); its reference maximum is raised only when a page's maximum
 * exceeds it by more than 2^8 (exact for any reference).
 *   ws: dllm_workspace_size(DLLM_OP_BLOCK_ATTENTION) bytes (currently 0). */
dllm_status dllm_block_attention(const dllm_layer_desc* desc, const dllm_batch* batch, const void* q_block,
                                 const dllm_cache* cache, void* o_full, float* lse, void* ws, size_t ws_bytes,
                                 void* stream);

/* Inner step, part 3 (LaCache §3.3.3 and Algorithm 1 with GenStep = False):
 * for every row r of U_b and head h, start from the cached state (m, l,
 * O~ = l o_pool)
 * of dllm_cache_build, stream only the B_b fresh block keys (read through
 * block_table at positions s_b .. s_b+B_b-1):
 *   m' = max_c S_rc, l' = sum_c exp(S_rc - m'), O' = sum_c exp(S_rc - m') v_c,
 *   m* = max(m, m'), l* = e^(m-m*) l + e^(m'-m*) l',
 *   O_r = (e^(m-m*) O~ + e^(m'-m*) O') / l*,  L_r = m* + ln l*,
 * and write O_r as bf16 to o_full row cu_seq[b] + r (and L_r to lse when
 * non-NULL).  The cache is read-only.
 *   ws: dllm_workspace_size(DLLM_OP_STATE_MERGE) bytes (currently 0). */
dllm_status dllm_state_merge(const dllm_layer_desc* desc, const dllm_batch* batch, const dllm_cache* cache,
                             void* o_full, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Inner step, parts 2 and 3 in one launch: the results of
 * dllm_block_attention followed by dllm_state_merge (both write disjoint rows
 * of o_full and lse), with the merge work filling the GPU while the block
 * attention finishes (no counterpart in the pages: a scheduling choice of
 * this library).
 *   ws: dllm_workspace_size(DLLM_OP_STEP_ATTENTION) bytes (currently 0). */
dllm_status dllm_step_attention(const dllm_layer_desc* desc, const dllm_batch* batch, const void* q_block,
                                const dllm_cache* cache, void* o_full, float* lse, void* ws, size_t ws_bytes,
                                void* stream);

/* Block-only epilogue after the layer stack (LaCache §3.4, the sampling
 * stage: the output is cut to the tokens of the current generation block;
 * Fast-dLLM "Block-wise Generation").  For the B_b rows of each current block
 * only (block row i of sequence b is row cu_seq[b] + s_b + i of h_full):
 *   x^ = RMSNorm(h) with gain final_gain (correctly rounded to bf16),
 *   logits = x^ W_lm^T (fp32 accumulation, W_lm bf16 [vocab][d_model]),
 *   and the softmax over the vocabulary, summarised per row as
 *   lse = log sum_v exp(logit_v), argmax = the lowest v with the largest
 *   logit, p_max = exp(logit_argmax - lse) (the confidence the sampler
 *   compares with its threshold),
 * written to lse, argmax, p_max (device [M] each, M = batch->total_block_rows,
 * packed by cu_block) and, when logits is non-NULL, the bf16 logits
 * [M][vocab].  d_model must be a multiple of 128 and vocab of 8.
 *   ws: dllm_lm_head_workspace_size bytes (the x^ rows and per-tile partial
 *   softmax statistics). */
dllm_status dllm_lm_head_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t vocab,
                                        size_t* bytes);
dllm_status dllm_block_lm_head(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t vocab,
                               const void* h_full, const void* final_gain, const void* w_lm, void* logits,
                               float* lse, int32_t* argmax, float* p_max, void* ws, size_t ws_bytes, void* stream);

/* The rest of the layer for the current blocks' rows, with the FFN in
 * per-group FP8 (LaCache §3.4 Mixed precision strategy, Eq. (7)-(8): a tensor
 * split into groups g is quantised as x' = clip(x / scale_g, -448, 448),
 * scale_g = max_g |x| / 448 (e4m3, round to nearest even), the quantisation
 * fused into the AddNorm before the gate-up linear and into the SwiGLU
 * before the down linear).  For the B_b rows of each current block
 * (block row i of sequence b: attention output row cu_seq[b] + s_b + i):
 *   h1 = x_block + O W_o^T                               (bf16 in, fp32 sum, bf16 h1)
 *   x2 = RMSNorm(h1) ffn_gain, quantised per row and 128 columns
 *   a  = SiLU(x2 W_gate^T) * (x2 W_up^T), quantised per row and 128 units
 *   y_block = h1 + a W_down^T                           (bf16)
 * where every e4m3 GEMM sums each group of 128 products in fp32 times the
 * product of its two scales.  Layouts (row-major):
 *   o_full:      bf16 [R][n_heads * head_dim] (dllm_block_attention's output)
 *   x_block:     bf16 [M][d_model], packed by cu_block (the layer's input rows)
 *   w_o:         bf16 [d_model][n_heads * head_dim]
 *   ffn_gain:    bf16 [d_model]
 *   w_gate_up:   e4m3 [2 d_ff][d_model]: row 2j is gate unit j, row 2j + 1 up unit j;
 *   w_gate_up_scale: fp32 [2 d_ff / 128][d_model / 128], one scale per 128 x 128 block
 *   w_down:      e4m3 [d_model][d_ff]; w_down_scale fp32 [d_model / 128][d_ff / 128]
 *   y_block:     bf16 [M][d_model], packed by cu_block
 * d_model and d_ff must be multiples of 128.
 *   ws: dllm_ffn_workspace_size bytes. */
dllm_status dllm_ffn_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t d_ff, size_t* bytes);
dllm_status dllm_block_ffn(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t d_ff, const void* o_full,
                           const void* x_block, const void* w_o, const void* ffn_gain, const void* w_gate_up,
                           const float* w_gate_up_scale, const void* w_down, const float* w_down_scale,
                           void* y_block, void* ws, size_t ws_bytes, void* stream);

/* Static description of a status code (never NULL). */
const char* dllm_status_string(dllm_status status);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* DLLM_H_ */
