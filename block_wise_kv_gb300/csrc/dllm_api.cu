// dllm_api.cu — the C ABI declared in include/dllm.h: host-side validation,
// workspace sizing and the launch sequence of each entry point.  Every check
// runs before the first launch, so a rejected call launches nothing.
#include <math.h>
#include <stdint.h>

#include "dllm.h"
#include "kernels.cuh"

using namespace dllm;

namespace {

constexpr int64_t kMaxRows = (int64_t{1} << 31) - 1;

bool aligned(const void* p, uintptr_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dllm_status check_desc(const dllm_layer_desc* d) {
  if (d == nullptr) return DLLM_ERR_INVALID_ARGUMENT;
  if (d->head_dim != 64 && d->head_dim != 128) return DLLM_ERR_UNSUPPORTED;
  if (d->page_size != kPage) return DLLM_ERR_UNSUPPORTED;
  if (d->d_model <= 0 || d->n_heads <= 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (d->d_model % 64 != 0) return DLLM_ERR_UNSUPPORTED;
  if ((static_cast<int64_t>(d->n_heads) * d->head_dim) % 128 != 0) return DLLM_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(d->n_heads) * d->head_dim * 3 > 65535 * 128) return DLLM_ERR_UNSUPPORTED;
  if (!(d->rope_theta > 0.f) || !isfinite(d->rope_theta)) return DLLM_ERR_INVALID_ARGUMENT;
  if (!(d->rms_eps >= 0.f) || !isfinite(d->rms_eps)) return DLLM_ERR_INVALID_ARGUMENT;
  if (!(d->softmax_scale >= 0.f) || !isfinite(d->softmax_scale)) return DLLM_ERR_INVALID_ARGUMENT;
  return DLLM_OK;
}

dllm_status check_batch(const dllm_batch* b) {
  if (b == nullptr || b->batch < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (b->batch == 0) return DLLM_OK;
  if (b->batch > 65535) return DLLM_ERR_UNSUPPORTED;
  if (!aligned(b->block_table, 4) || !aligned(b->seq_len, 4) || !aligned(b->block_start, 4) ||
      !aligned(b->block_len, 4) || !aligned(b->cu_block, 4) || !aligned(b->cu_seq, 4))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (b->error_flag != nullptr && !aligned(b->error_flag, 4)) return DLLM_ERR_INVALID_ARGUMENT;
  if (b->max_pages_per_seq < 1 || b->max_seq_len < 1 || b->max_block_len < 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (b->max_block_len > b->max_seq_len) return DLLM_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(b->max_pages_per_seq) * kPage < b->max_seq_len) return DLLM_ERR_INVALID_ARGUMENT;
  if (b->max_seq_len > 65535 * kPage) return DLLM_ERR_UNSUPPORTED;
  if (b->total_block_rows < 0 || b->total_seq_rows < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(b->total_block_rows) > static_cast<int64_t>(b->batch) * b->max_block_len)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(b->total_seq_rows) > static_cast<int64_t>(b->batch) * b->max_seq_len)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (b->total_block_rows > b->total_seq_rows) return DLLM_ERR_INVALID_ARGUMENT;
  return DLLM_OK;
}

dllm_status check_cache(const dllm_cache* c, const dllm_layer_desc* d, bool need_q, bool need_state) {
  if (c == nullptr || c->num_pages < 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (static_cast<int64_t>(c->num_pages) * d->n_heads * kPage > kMaxRows) return DLLM_ERR_UNSUPPORTED;
  if (!aligned(c->k_pool, 16) || !aligned(c->v_pool, 16)) return DLLM_ERR_INVALID_ARGUMENT;
  if (need_q && !aligned(c->q_pool, 16)) return DLLM_ERR_INVALID_ARGUMENT;
  if (need_state && (!aligned(c->m_pool, 16) || !aligned(c->l_pool, 16) || !aligned(c->o_pool, 16)))
    return DLLM_ERR_INVALID_ARGUMENT;
  return DLLM_OK;
}

// The prefix state pools: all unset (0), all set and aligned (1), else invalid (-1).
int pre_pools(const dllm_cache* c) {
  if (c->m_pre == nullptr && c->l_pre == nullptr && c->o_pre == nullptr) return 0;
  if (!aligned(c->m_pre, 16) || !aligned(c->l_pre, 16) || !aligned(c->o_pre, 16)) return -1;
  return 1;
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

BatchArgs batch_args(const dllm_batch* b, const dllm_cache* c) {
  BatchArgs a;
  a.block_table = b->block_table;
  a.seq_len = b->seq_len;
  a.block_start = b->block_start;
  a.block_len = b->block_len;
  a.cu_block = b->cu_block;
  a.cu_seq = b->cu_seq;
  a.err = b->error_flag;
  a.batch = b->batch;
  a.max_pages = b->max_pages_per_seq;
  a.num_pages = c->num_pages;
  a.max_block_len = b->max_block_len;
  a.max_seq_len = b->max_seq_len;
  a.total_block_rows = b->total_block_rows;
  a.total_seq_rows = b->total_seq_rows;
  return a;
}

float softmax_scale(const dllm_layer_desc* d) {
  return d->softmax_scale > 0.f ? d->softmax_scale : static_cast<float>(1.0 / sqrt(static_cast<double>(d->head_dim)));
}

AttnArgs attn_args(const dllm_layer_desc* d, const dllm_batch* b, const dllm_cache* c) {
  AttnArgs a;
  a.bt = batch_args(b, c);
  a.q_block = nullptr;
  a.k_pool = c->k_pool;
  a.v_pool = c->v_pool;
  a.q_pool = c->q_pool;
  a.m_pool = c->m_pool;
  a.l_pool = c->l_pool;
  a.o_pool = c->o_pool;
  a.o_full = nullptr;
  a.lse = nullptr;
  a.n_heads = d->n_heads;
  a.head_dim = d->head_dim;
  a.scale_log2 = softmax_scale(d) * 1.4426950408889634f;
  a.m_pre = nullptr;
  a.l_pre = nullptr;
  a.o_pre = nullptr;
  a.prev_start = nullptr;
  return a;
}

AttnPlan plan_of(const dllm_layer_desc* d, const dllm_batch* b, bool block, bool merge) {
  return attn_plan(b->batch, d->n_heads, d->head_dim, b->max_seq_len, b->max_block_len, b->total_seq_rows,
                   b->total_block_rows, device_sms(), block, merge);
}



QkvArgs qkv_args(const dllm_layer_desc* d, const dllm_batch* b, const dllm_cache* c, const float* rope,
                 int32_t rope_max_pos, int mode, int n_tok) {
  QkvArgs a;
  a.bt = batch_args(b, c);
  a.k_pool = c->k_pool;
  a.v_pool = c->v_pool;
  a.q_pool = c->q_pool;
  a.q_block = nullptr;
  a.rope = rope;
  a.rope_max_pos = rope_max_pos;
  a.n_heads = d->n_heads;
  a.head_dim = d->head_dim;
  a.d_model = d->d_model;
  a.n_tok = n_tok;
  a.mode = mode;
  a.x = nullptr;
  a.gain = nullptr;
  a.rms_eps = d->rms_eps;
  a.xhat = nullptr;
  a.inv = nullptr;
  a.norm_ctr = nullptr;
  a.partials = nullptr;
  a.counters = nullptr;
  a.max_contrib = 0;
  return a;
}

// Point the projection at its workspace: the counters (RMSNorm row claims,
// then the stream-K tile arrivals), the per-row RMSNorm scales, the x^ rows,
// and (stream-K) the fp32 partial tiles.
void bind_workspace(QkvArgs* a, const QkvPlan& plan, void* ws) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  a->norm_ctr = reinterpret_cast<int32_t*>(base);
  a->inv = reinterpret_cast<float2*>(base + plan.inv_offset);
  a->xhat = base + plan.xhat_offset;
  if (!plan.streamk) return;
  a->counters = reinterpret_cast<int32_t*>(base) + kQkvNormCounters;
  a->partials = reinterpret_cast<float*>(base + plan.part_offset);
  a->max_contrib = plan.max_contrib;
}

dllm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DLLM_OK : DLLM_ERR_CUDA; }

#define DLLM_TRY(expr)                     \
  do {                                     \
    const dllm_status s_ = (expr);         \
    if (s_ != DLLM_OK) return s_;          \
  } while (0)

#define DLLM_CUDA_TRY(expr)                \
  do {                                     \
    const cudaError_t e_ = (expr);         \
    if (e_ != cudaSuccess) return DLLM_ERR_CUDA; \
  } while (0)

}  // namespace

extern "C" {

dllm_status dllm_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t op, size_t* bytes) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (bytes == nullptr) return DLLM_ERR_INVALID_ARGUMENT;
  switch (op) {
    case DLLM_OP_CACHE_BUILD:
      *bytes = batch->batch > 0 && batch->total_seq_rows > 0
                   ? qkv_plan(batch->total_seq_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms())
                         .total_bytes
                   : 0;
      return DLLM_OK;
    case DLLM_OP_BLOCK_QKV_ROPE_WRITE:
      *bytes = batch->batch > 0 && batch->total_block_rows > 0
                   ? qkv_plan(batch->total_block_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms())
                         .total_bytes
                   : 0;
      return DLLM_OK;
    case DLLM_OP_BLOCK_ATTENTION:
      *bytes = batch->batch > 0 && batch->total_block_rows > 0 ? plan_of(desc, batch, true, false).total_bytes : 0;
      return DLLM_OK;
    case DLLM_OP_STEP_ATTENTION:
      *bytes = batch->batch > 0 && batch->total_block_rows > 0 ? plan_of(desc, batch, true, true).total_bytes : 0;
      return DLLM_OK;
    case DLLM_OP_STATE_MERGE:
      *bytes = 0;
      return DLLM_OK;
    case DLLM_OP_CACHE_ADVANCE:  // `batch` is the decoded blocks': the projection of their rows
      *bytes = batch->batch > 0 && batch->total_block_rows > 0
                   ? qkv_plan(batch->total_block_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms())
                         .total_bytes
                   : 0;
      return DLLM_OK;
    default:
      return DLLM_ERR_INVALID_ARGUMENT;
  }
}

dllm_status dllm_qkv_weight_packed_bytes(const dllm_layer_desc* desc, size_t* bytes) {
  if (bytes == nullptr) return DLLM_ERR_INVALID_ARGUMENT;
  DLLM_TRY(check_desc(desc));
  *bytes = qkv_packed_bytes(desc->d_model, desc->n_heads, desc->head_dim);
  return DLLM_OK;
}

dllm_status dllm_qkv_weight_pack(const dllm_layer_desc* desc, const void* w_qkv, void* w_packed, void* stream) {
  DLLM_TRY(check_desc(desc));
  if (!aligned(w_qkv, 16) || !aligned(w_packed, 16))
    return DLLM_ERR_INVALID_ARGUMENT;
  const size_t in_bytes = static_cast<size_t>(3) * desc->n_heads * desc->head_dim * desc->d_model * 2;
  const size_t out_bytes = qkv_packed_bytes(desc->d_model, desc->n_heads, desc->head_dim);
  const uintptr_t a = reinterpret_cast<uintptr_t>(w_qkv), b = reinterpret_cast<uintptr_t>(w_packed);
  if (a < b + out_bytes && b < a + in_bytes) return DLLM_ERR_INVALID_ARGUMENT;  // overlapping
  DLLM_CUDA_TRY(launch_qkv_pack(w_qkv, w_packed, 3 * desc->n_heads * desc->head_dim, desc->d_model,
                                static_cast<cudaStream_t>(stream)));
  return DLLM_OK;
}

dllm_status dllm_rope_table_build(const dllm_layer_desc* desc, int32_t max_pos, float* rope_table, void* stream) {
  DLLM_TRY(check_desc(desc));
  if (max_pos < 1 || !aligned(rope_table, 8)) return DLLM_ERR_INVALID_ARGUMENT;
  return cuda_status(launch_rope_table(rope_table, max_pos, desc->head_dim, static_cast<double>(desc->rope_theta),
                                       static_cast<cudaStream_t>(stream)));
}

dllm_status dllm_cache_build(const dllm_layer_desc* desc, const dllm_batch* batch, const void* x_full,
                             const void* rms_gain, const void* w_packed, const float* rope_table, int32_t rope_max_pos,
                             const dllm_cache* cache, void* ws, size_t ws_bytes, void* stream) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (batch->batch == 0 || batch->total_seq_rows == 0) return DLLM_OK;
  DLLM_TRY(check_cache(cache, desc, true, true));
  const int pre = pre_pools(cache);
  if (pre < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (!aligned(x_full, 16) || !aligned(rms_gain, 16) || !aligned(w_packed, 16) || !aligned(rope_table, 8))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (rope_max_pos < batch->max_seq_len) return DLLM_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  DLLM_TRY(dllm_workspace_size(desc, batch, DLLM_OP_CACHE_BUILD, &need));
  if (ws_bytes < need) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const BatchArgs bt = batch_args(batch, cache);
  const QkvPlan plan = qkv_plan(batch->total_seq_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms());
  QkvArgs qa = qkv_args(desc, batch, cache, rope_table, rope_max_pos, kModeBoundary, batch->total_seq_rows);
  qa.x = x_full;
  qa.gain = rms_gain;
  bind_workspace(&qa, plan, ws);
  DLLM_CUDA_TRY(launch_zero_tails(bt, cache->k_pool, cache->v_pool, cache->q_pool, desc->n_heads, desc->head_dim, s));
  DLLM_CUDA_TRY(launch_qkv_gemm(w_packed, qa, plan, s));
  AttnArgs aa = attn_args(desc, batch, cache);
  if (pre) {
    aa.m_pre = cache->m_pre;
    aa.l_pre = cache->l_pre;
    aa.o_pre = cache->o_pre;
  }
  DLLM_CUDA_TRY(launch_rows_attention(aa, pre ? kRowsStatePre : kRowsState, device_sms(), s));
  return DLLM_OK;
}

dllm_status dllm_cache_advance(const dllm_layer_desc* desc, const dllm_batch* batch, const dllm_batch* decoded,
                               const void* x_decoded, const void* rms_gain, const void* w_packed,
                               const float* rope_table, int32_t rope_max_pos, const dllm_cache* cache, void* ws,
                               size_t ws_bytes, void* stream) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  DLLM_TRY(check_batch(decoded));
  // the decoded blocks describe the same sequences, through the same metadata
  if (decoded->batch != batch->batch || decoded->block_table != batch->block_table ||
      decoded->seq_len != batch->seq_len || decoded->cu_seq != batch->cu_seq ||
      decoded->max_pages_per_seq != batch->max_pages_per_seq || decoded->total_seq_rows != batch->total_seq_rows ||
      decoded->max_seq_len != batch->max_seq_len)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (batch->batch == 0 || batch->total_seq_rows == 0) return DLLM_OK;
  DLLM_TRY(check_cache(cache, desc, true, true));
  if (pre_pools(cache) != 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (!aligned(x_decoded, 16) || !aligned(rms_gain, 16) || !aligned(w_packed, 16) || !aligned(rope_table, 8))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (rope_max_pos < batch->max_seq_len) return DLLM_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  DLLM_TRY(dllm_workspace_size(desc, decoded, DLLM_OP_CACHE_ADVANCE, &need));
  if (ws_bytes < need) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // the decoded rows: q, k, v into the pools
  if (decoded->total_block_rows > 0) {
    const QkvPlan plan =
        qkv_plan(decoded->total_block_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms());
    QkvArgs qa = qkv_args(desc, decoded, cache, rope_table, rope_max_pos, kModeRows, decoded->total_block_rows);
    qa.x = x_decoded;
    qa.gain = rms_gain;
    bind_workspace(&qa, plan, ws);
    DLLM_CUDA_TRY(launch_qkv_gemm(w_packed, qa, plan, s));
  }
  // the prefix state extended (rows kept) or rebuilt (decoded rows), then the state over U
  AttnArgs aa = attn_args(desc, batch, cache);
  aa.m_pre = cache->m_pre;
  aa.l_pre = cache->l_pre;
  aa.o_pre = cache->o_pre;
  aa.prev_start = decoded->block_start;
  DLLM_CUDA_TRY(launch_rows_attention(aa, kRowsAdvOld, device_sms(), s));
  DLLM_CUDA_TRY(launch_rows_attention(aa, kRowsAdvNew, device_sms(), s));
  return DLLM_OK;
}

dllm_status dllm_block_qkv_rope_write(const dllm_layer_desc* desc, const dllm_batch* batch, const void* x_block,
                                      const void* rms_gain, const void* w_packed, const float* rope_table,
                                      int32_t rope_max_pos, const dllm_cache* cache, void* q_block, void* ws,
                                      size_t ws_bytes, void* stream) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (batch->batch == 0 || batch->total_block_rows == 0) return DLLM_OK;
  DLLM_TRY(check_cache(cache, desc, false, false));
  if (!aligned(x_block, 16) || !aligned(rms_gain, 16) || !aligned(w_packed, 16) || !aligned(rope_table, 8) ||
      !aligned(q_block, 16))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (rope_max_pos < batch->max_seq_len) return DLLM_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  DLLM_TRY(dllm_workspace_size(desc, batch, DLLM_OP_BLOCK_QKV_ROPE_WRITE, &need));
  if (ws_bytes < need) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const QkvPlan plan = qkv_plan(batch->total_block_rows, desc->d_model, desc->n_heads, desc->head_dim, device_sms());
  QkvArgs qa = qkv_args(desc, batch, cache, rope_table, rope_max_pos, kModeBlock, batch->total_block_rows);
  qa.q_block = q_block;
  qa.x = x_block;
  qa.gain = rms_gain;
  bind_workspace(&qa, plan, ws);
  DLLM_CUDA_TRY(launch_qkv_gemm(w_packed, qa, plan, s));
  return DLLM_OK;
}

namespace {
// The common part of the three attention calls: validate, bind the workspace, launch.
dllm_status attention_call(const dllm_layer_desc* desc, const dllm_batch* batch, const void* q_block,
                           const dllm_cache* cache, void* o_full, float* lse, void* ws, size_t ws_bytes, void* stream,
                           bool block, bool merge) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (batch->batch == 0 || batch->total_seq_rows == 0) return DLLM_OK;
  if (block && batch->total_block_rows == 0) block = false;
  if (!block && !merge) return DLLM_OK;
  // Blocks of at most one page run on the fused streaming kernel; longer blocks (the
  // prefix-only cache mode, where the block is everything after the prefix) on the
  // 128-row query-tile kernel, one launch per part.
  const bool wide = batch->max_block_len > kPage;
  if (!wide && !attn_batch_supported(batch->batch)) return DLLM_ERR_UNSUPPORTED;
  DLLM_TRY(check_cache(cache, desc, merge, merge));
  if (block && !aligned(q_block, 16)) return DLLM_ERR_INVALID_ARGUMENT;
  if (!aligned(o_full, 16)) return DLLM_ERR_INVALID_ARGUMENT;
  if (lse != nullptr && !aligned(lse, 4)) return DLLM_ERR_INVALID_ARGUMENT;
  const AttnPlan plan = plan_of(desc, batch, block, merge);
  if (ws_bytes < plan.total_bytes) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (plan.total_bytes > 0 && !aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  AttnArgs aa = attn_args(desc, batch, cache);
  aa.q_block = q_block;
  aa.o_full = o_full;
  aa.lse = lse;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (wide) {
    if (block) DLLM_CUDA_TRY(launch_rows_attention(aa, kRowsBlock, device_sms(), s));
    if (merge) DLLM_CUDA_TRY(launch_rows_attention(aa, kRowsMerge, device_sms(), s));
    return DLLM_OK;
  }
  DLLM_CUDA_TRY(launch_step_attention(aa, plan, s));
  return DLLM_OK;
}
}  // namespace

dllm_status dllm_block_attention(const dllm_layer_desc* desc, const dllm_batch* batch, const void* q_block,
                                 const dllm_cache* cache, void* o_full, float* lse, void* ws, size_t ws_bytes,
                                 void* stream) {
  return attention_call(desc, batch, q_block, cache, o_full, lse, ws, ws_bytes, stream, true, false);
}

dllm_status dllm_state_merge(const dllm_layer_desc* desc, const dllm_batch* batch, const dllm_cache* cache,
                             void* o_full, float* lse, void* ws, size_t ws_bytes, void* stream) {
  return attention_call(desc, batch, nullptr, cache, o_full, lse, ws, ws_bytes, stream, false, true);
}

dllm_status dllm_step_attention(const dllm_layer_desc* desc, const dllm_batch* batch, const void* q_block,
                                const dllm_cache* cache, void* o_full, float* lse, void* ws, size_t ws_bytes,
                                void* stream) {
  return attention_call(desc, batch, q_block, cache, o_full, lse, ws, ws_bytes, stream, true, true);
}

dllm_status dllm_lm_head_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t vocab,
                                        size_t* bytes) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (bytes == nullptr || vocab < 1) return DLLM_ERR_INVALID_ARGUMENT;
  *bytes = batch->batch > 0 && batch->total_block_rows > 0
               ? lm_head_workspace_bytes(batch->total_block_rows, desc->d_model, vocab)
               : 0;
  return DLLM_OK;
}

dllm_status dllm_block_lm_head(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t vocab,
                               const void* h_full, const void* final_gain, const void* w_lm, void* logits,
                               float* lse, int32_t* argmax, float* p_max, void* ws, size_t ws_bytes, void* stream) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (vocab < 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (desc->d_model % 128 != 0 || vocab % 8 != 0) return DLLM_ERR_UNSUPPORTED;
  if (batch->batch == 0 || batch->total_block_rows == 0) return DLLM_OK;
  if (!aligned(h_full, 16) || !aligned(final_gain, 16) || !aligned(w_lm, 16) || !aligned(lse, 4) ||
      !aligned(argmax, 4) || !aligned(p_max, 4))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (logits != nullptr && !aligned(logits, 16)) return DLLM_ERR_INVALID_ARGUMENT;
  size_t need = 0;
  DLLM_TRY(dllm_lm_head_workspace_size(desc, batch, vocab, &need));
  if (ws_bytes < need) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  LmArgs a;
  dllm_cache none = {};
  none.num_pages = 1;
  a.bt = batch_args(batch, &none);
  a.h = h_full;
  a.gain = final_gain;
  a.logits = logits;
  a.lse = lse;
  a.argmax = argmax;
  a.p_max = p_max;
  a.n_rows = batch->total_block_rows;
  a.d_model = desc->d_model;
  a.vocab = vocab;
  a.rms_eps = desc->rms_eps;
  lm_bind_workspace(&a, ws);
  DLLM_CUDA_TRY(launch_lm_head(w_lm, a, device_sms(), static_cast<cudaStream_t>(stream)));
  return DLLM_OK;
}

dllm_status dllm_ffn_workspace_size(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t d_ff,
                                    size_t* bytes) {
  DLLM_TRY(check_desc(desc));
  DLLM_TRY(check_batch(batch));
  if (bytes == nullptr || d_ff < 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (desc->d_model % 128 != 0 || d_ff % 128 != 0) return DLLM_ERR_UNSUPPORTED;
  *bytes = batch->batch > 0 && batch->total_block_rows > 0
               ? ffn_workspace_bytes(batch->total_block_rows, desc->d_model, desc->n_heads * desc->head_dim, d_ff,
                                     device_sms())
               : 0;
  return DLLM_OK;
}

dllm_status dllm_block_ffn(const dllm_layer_desc* desc, const dllm_batch* batch, int32_t d_ff, const void* o_full,
                           const void* x_block, const void* w_o, const void* ffn_gain, const void* w_gate_up,
                           const float* w_gate_up_scale, const void* w_down, const float* w_down_scale,
                           void* y_block, void* ws, size_t ws_bytes, void* stream) {
  size_t need = 0;
  DLLM_TRY(dllm_ffn_workspace_size(desc, batch, d_ff, &need));
  if (batch->batch == 0 || batch->total_block_rows == 0) return DLLM_OK;
  if (!aligned(o_full, 16) || !aligned(x_block, 16) || !aligned(w_o, 16) || !aligned(ffn_gain, 16) ||
      !aligned(w_gate_up, 16) || !aligned(w_gate_up_scale, 4) || !aligned(w_down, 16) || !aligned(w_down_scale, 4) ||
      !aligned(y_block, 16))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (ws_bytes < need) return DLLM_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(ws, 256)) return DLLM_ERR_INVALID_ARGUMENT;
  FfnArgs a = {};
  dllm_cache none = {};
  none.num_pages = 1;
  a.bt = batch_args(batch, &none);
  a.o_full = o_full;
  a.x_block = x_block;
  a.gain2 = ffn_gain;
  a.y = y_block;
  a.n_rows = batch->total_block_rows;
  a.d_model = desc->d_model;
  a.hd = desc->n_heads * desc->head_dim;
  a.d_ff = d_ff;
  a.rms_eps = desc->rms_eps;
  FfnWeights w;
  w.w_o = w_o;
  w.w_gu = w_gate_up;
  w.gu_scale = w_gate_up_scale;
  w.w_down = w_down;
  w.down_scale = w_down_scale;
  DLLM_CUDA_TRY(launch_ffn(a, w, ws, device_sms(), static_cast<cudaStream_t>(stream)));
  return DLLM_OK;
}

const char* dllm_status_string(dllm_status status) {
  switch (status) {
    case DLLM_OK:
      return "ok";
    case DLLM_ERR_INVALID_ARGUMENT:
      return "invalid argument";
    case DLLM_ERR_UNSUPPORTED:
      return "unsupported shape or configuration";
    case DLLM_ERR_WORKSPACE_TOO_SMALL:
      return "workspace too small";
    case DLLM_ERR_CUDA:
      return "CUDA error";
    case DLLM_ERR_TIMEOUT:
      return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
