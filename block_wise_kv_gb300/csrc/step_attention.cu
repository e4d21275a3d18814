// step_attention.cu — the attention part of an inner denoising step in one
// launch (sm_103a): the block rows' attention over every key of their
// sequence and the FACache merge of every invariant row.
//
//   block items   (sequence b, head h, chunk c): the block queries of (b, h)
//                 (<= 64 rows) against the keys of chunk_pages consecutive
//                 pages, read page by page through the block table (Fast-dLLM
//                 DualCache: [prefix KV | fresh block KV | suffix KV]).  With
//                 several chunks, each CTA leaves its partial online-softmax
//                 state in the workspace and the last chunk to arrive merges
//                 them exactly (LaCache Eq. (2)-(6) applied to states).
//   merge items   (sequence b, head h, query page p): for the rows of U in
//                 page p, the cached state (m, l, O~) merged with the fresh
//                 partial state over the block keys (LaCache Eq. (2)-(6);
//                 Algorithm 1 with GenStep = False).
//
// One grid holds both kinds, block items first: they are the longer ones, so
// they start first, and merge CTAs fill every SM slot as soon as one frees
// (no second kernel waiting for the first to drain).  Every tile that can be
// is moved by TMA (128-byte swizzle): the block queries through a 3-D tensor
// map over q_block, K/V pages, the query page and the fp32 O~ page.  The
// QK^T / PV contractions of each warp's 16 query rows run on mma.sync
// m16n8k16 (bf16 in, fp32 accumulate); row max and sum use quad shuffles.
//
// Programmatic dependent launch: barrier setup overlaps the tail of the
// preceding kernel; every read of data it may write comes after
// griddepcontrol.wait.
#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

template <int D>
struct StepCfg {
  static constexpr int TB = tile_bytes<D>();
  static constexpr int kStages = 2;  // K/V page pairs in flight per block item
  static constexpr int kBlockSmem = TB * (1 + 2 * kStages);
  static constexpr int kMergeSmem = TB * 3 + 64 * D * 4;  // q page | K_C | V_C | O~ page (fp32)
  static constexpr int kSmem = (kBlockSmem > kMergeSmem ? kBlockSmem : kMergeSmem) + 1024;
  static constexpr int kOStride = D + 8;  // padded fp32 row of the per-warp partials
  static constexpr int kPartStride = D + 4;  // workspace partial row: D accumulators, then (m, l)
  static_assert(64 * kOStride * 4 <= kBlockSmem, "per-warp partials must fit in the drained ring");
};

constexpr int kThreads = 160;  // warps 0-3 compute, warp 4 streams tiles

// ----------------------------------------------------------- block item
template <int D>
__device__ __forceinline__ void block_item(const CUtensorMap* tm_qb, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                           const AttnArgs& a, uint8_t* smem, uint64_t* full_bar, uint64_t* empty_bar,
                                           uint64_t* q_bar, float* comb_m, float* comb_l, int* flag, long long idx) {
  constexpr int TB = StepCfg<D>::TB;
  constexpr int NST = StepCfg<D>::kStages;
  constexpr int OS = StepCfg<D>::kOStride;
  constexpr int PS = StepCfg<D>::kPartStride;
  constexpr int C4 = D / 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads, S = a.n_chunks;
  const int c = static_cast<int>(idx % S), h = static_cast<int>((idx / S) % H), b = static_cast<int>(idx / (S * H));
  const SeqMeta sm = load_meta(bt, b);
  if (!sm.ok) {
    if (threadIdx.x == 0 && c == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int npages = (sm.nb + kPage - 1) / kPage;
  const int n_chunks_b = (npages + a.chunk_pages - 1) / a.chunk_pages;
  const int p0 = c * a.chunk_pages, p1 = min(npages, p0 + a.chunk_pages);
  if (p0 >= npages) return;  // this sequence needs fewer chunks
  const int my = p1 - p0;
  const int RG = (sm.bb + 15) / 16;  // 16-row groups of block queries
  const int KS = 4 / RG;             // key slices per page
  const bool active = warp < 4 && warp < RG * KS;
  const int rg = warp % RG, ks = warp / RG;
  uint8_t* q_tile = smem;
  uint8_t* kv = smem + TB;
  float* comb_o = reinterpret_cast<float*>(smem);  // [64][OS] after the page loop

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 4);
    }
    mbar_init(q_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  WarpAttn<D> st;
  st.init();
  if (warp == 4) {
    if (lane == 0) {  // ---- TMA producer: the block queries, then the chunk's K/V pages
      mbar_arrive_expect_tx(q_bar, TB);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) tma_load_3d(q_tile + hf * 8192, tm_qb, q_bar, hf * 64, h, sm.cub);
      int issued = 0;
      for (int i = 0; i < my; ++i) {
        const int s = i % NST;
        const uint32_t ph = (i / NST) & 1;
        if (i >= NST && !mbar_wait(&empty_bar[s], ph ^ 1)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        const int pg = page_of(bt, b, p0 + i);
        uint8_t* kt = kv + s * 2 * TB;
        const int y = (pg * H + h) * kPage;
        mbar_arrive_expect_tx(&full_bar[s], 2 * TB);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_2d(kt + hf * 8192, tm_k, &full_bar[s], hf * 64, y);
          tma_load_2d(kt + TB + hf * 8192, tm_v, &full_bar[s], hf * 64, y);
        }
        ++issued;
      }
      // every issued copy has landed before the buffers are reused or the CTA exits
      for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % NST], (i / NST) & 1)) report_error(bt.err, kErrTimeout);
      if (!mbar_wait(q_bar, 0)) report_error(bt.err, kErrTimeout);
    }
  } else {  // ---- compute warps
    const bool q_ok = mbar_wait(q_bar, 0);
    if (!q_ok) report_error(bt.err, kErrTimeout);
    uint32_t qf[D / 16][4];
    if (active) load_q_frags<D>(qf, smem_u32(q_tile), rg * 16, lane);
    const int nk = 64 / KS, key0 = ks * nk;
    for (int i = 0; i < my && q_ok; ++i) {
      const int s = i % NST;
      const uint32_t ph = (i / NST) & 1;
      if (!mbar_wait(&full_bar[s], ph)) {
        report_error(bt.err, kErrTimeout);
        break;
      }
      if (active) {
        const uint32_t kt = smem_u32(kv + s * 2 * TB), vt = kt + TB;
        const int base = (p0 + i) * kPage;
        const int nb = sm.nb;
        auto valid = [base, nb](int key) { return base + key < nb; };
        if (KS == 1)
          attend<D, 64>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
        else if (KS == 2)
          attend<D, 32>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
        else
          attend<D, 16>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }
  __syncthreads();  // every page consumed and every copy landed: the ring holds the per-warp partials

  if (active) {
    st.reduce_l();
    const int g = lane >> 2, t = lane & 3;
    const int slot0 = ks * RG * 16 + rg * 16 + g, slot1 = slot0 + 8;
    if (t == 0) {
      comb_m[slot0] = st.m[0];
      comb_l[slot0] = st.l[0];
      comb_m[slot1] = st.m[1];
      comb_l[slot1] = st.l[1];
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(comb_o + slot0 * OS + 8 * n + 2 * t) = make_float2(st.o[n][0], st.o[n][1]);
      *reinterpret_cast<float2*>(comb_o + slot1 * OS + 8 * n + 2 * t) = make_float2(st.o[n][2], st.o[n][3]);
    }
  }
  __syncthreads();

  __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
  float* mypart = a.part + ((static_cast<size_t>(b) * H + h) * S + c) * 64 * PS;
  // ---- combine the KS key-slice partials of each row; finish the row (one
  // chunk) or leave the chunk's state in the workspace
  for (int item = threadIdx.x; item < sm.bb * C4; item += kThreads) {
    const int i = item / C4, col = (item % C4) * 4;
    float M = neg_inf();
    for (int q = 0; q < KS; ++q) M = fmaxf(M, comb_m[q * RG * 16 + i]);
    const float Mu = M == neg_inf() ? 0.f : M;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < KS; ++q) {
      const int slot = q * RG * 16 + i;
      const float w = fast_exp2(comb_m[slot] - Mu);
      L += w * comb_l[slot];
      const float4 ov = *reinterpret_cast<const float4*>(comb_o + slot * OS + col);
      acc.x += w * ov.x;
      acc.y += w * ov.y;
      acc.z += w * ov.z;
      acc.w += w * ov.w;
    }
    if (n_chunks_b == 1) {
      const float inv = 1.f / L;
      const size_t orow = static_cast<size_t>(sm.cus + sm.sb + i) * H + h;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(of + orow * D + col) = pk;
      if (a.lse != nullptr && col == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
    } else {
      *reinterpret_cast<float4*>(mypart + i * PS + col) = acc;
      if (col == 0) *reinterpret_cast<float2*>(mypart + i * PS + D) = make_float2(M, L);
    }
  }
  if (n_chunks_b == 1) return;

  // ---- count this chunk; the last of the sequence's chunks merges them all
  __syncthreads();  // the chunk's partial rows are written ...
  int32_t* counter = a.counters + static_cast<size_t>(b) * H + h;
  if (threadIdx.x == 0) {
    __threadfence();  // ... and (cumulatively) visible GPU-wide before the arrival is counted
    *flag = atomicAdd(counter, 1) == n_chunks_b - 1;
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  const float* part0 = a.part + (static_cast<size_t>(b) * H + h) * S * 64 * PS;
  for (int item = threadIdx.x; item < sm.bb * C4; item += kThreads) {
    const int i = item / C4, col = (item % C4) * 4;
    float M = neg_inf();
    for (int q = 0; q < n_chunks_b; ++q) M = fmaxf(M, __ldcg(part0 + (q * 64 + i) * PS + D));
    const float Mu = M == neg_inf() ? 0.f : M;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < n_chunks_b; ++q) {
      const float* pr = part0 + (q * 64 + i) * PS;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(pr + D));
      const float w = fast_exp2(ml.x - Mu);
      L += w * ml.y;
      const float4 ov = __ldcg(reinterpret_cast<const float4*>(pr + col));
      acc.x += w * ov.x;
      acc.y += w * ov.y;
      acc.z += w * ov.z;
      acc.w += w * ov.w;
    }
    const float inv = 1.f / L;
    const size_t orow = static_cast<size_t>(sm.cus + sm.sb + i) * H + h;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(of + orow * D + col) = pk;
    if (a.lse != nullptr && col == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
  }
  if (threadIdx.x == 0) *counter = 0;  // ready for the next call
}

// ----------------------------------------------------------- merge item
template <int D>
__device__ __forceinline__ void merge_item(const CUtensorMap* tm_q, const CUtensorMap* tm_o, const AttnArgs& a,
                                           uint8_t* smem, uint64_t* t_bar, float* m_s, float* l_s, long long idx,
                                           int max_pages) {
  constexpr int TB = StepCfg<D>::TB;
  uint8_t* q_tile = smem;  // later: staging of the bf16 output rows
  uint8_t* kc_tile = smem + TB;
  uint8_t* vc_tile = smem + 2 * TB;
  uint8_t* o_tile = smem + 3 * TB;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  const int qp = static_cast<int>(idx % max_pages), h = static_cast<int>((idx / max_pages) % H),
            b = static_cast<int>(idx / (static_cast<long long>(max_pages) * H));
  const SeqMeta sm = load_meta(bt, b);
  if (!sm.ok) {
    if (threadIdx.x == 0 && qp == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int npages = (sm.nb + kPage - 1) / kPage;
  if (qp >= npages) return;
  const int r_lo = qp * kPage, r_hi = min(sm.nb, r_lo + kPage);
  const int c_lo = sm.sb, c_hi = sm.sb + sm.bb;
  if (!((r_lo < c_lo) || (r_hi > c_hi))) return;  // no row of U in this page
  const int pgq = page_of(bt, b, qp);
  const size_t srow0 = (static_cast<size_t>(pgq) * H + h) * kPage;

  if (threadIdx.x == 0) {
    mbar_init(t_bar, 1);
    fence_barrier_init();
    // queries and cached O~ of the page's rows
    mbar_arrive_expect_tx(t_bar, TB + 64 * D * 4);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(q_tile + hf * 8192, tm_q, t_bar, hf * 64, static_cast<int>(srow0));
#pragma unroll
    for (int j = 0; j < D / 32; ++j) tma_load_2d(o_tile + j * 8192, tm_o, t_bar, j * 32, static_cast<int>(srow0));
  }
  // cached m, l of the page's rows; block keys/values gathered through the table
  if (threadIdx.x < 64) {
    m_s[threadIdx.x] = a.m_pool[srow0 + threadIdx.x];
    l_s[threadIdx.x] = a.l_pool[srow0 + threadIdx.x];
  }
  const int nkc = (sm.bb + 15) & ~15;
  {
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
    for (int e = threadIdx.x; e < nkc * (D / 8); e += kThreads) {
      const int cc = e / (D / 8), ch = e % (D / 8);
      uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
      if (cc < sm.bb) {
        const int pos = c_lo + cc;
        const int pg = page_of(bt, b, pos / kPage);
        const size_t off = ((static_cast<size_t>(pg) * H + h) * kPage + (pos % kPage)) * D;
        kv4 = __ldg(reinterpret_cast<const uint4*>(kp + off) + ch);
        vv4 = __ldg(reinterpret_cast<const uint4*>(vp + off) + ch);
      }
      *reinterpret_cast<uint4*>(kc_tile + tile_off(cc, ch)) = kv4;
      *reinterpret_cast<uint4*>(vc_tile + tile_off(cc, ch)) = vv4;
    }
  }
  __syncthreads();  // also orders the barrier initialisation before the waits below
  const bool loaded = mbar_wait(t_bar, 0);
  if (!loaded) report_error(bt.err, kErrTimeout);
  if (warp >= 4) return;  // the compute below is the 4 warps' 64 rows

  // fresh partial state over the block keys (Eq. (2)-(6) from the empty state)
  WarpAttn<D> st;
  st.init();
  uint32_t qf[D / 16][4];
  load_q_frags<D>(qf, smem_u32(q_tile), warp * 16, lane);
  const uint32_t kt = smem_u32(kc_tile), vt = smem_u32(vc_tile);
  const int bb = sm.bb;
  auto valid = [bb](int key) { return key < bb; };
  if (nkc == 16)
    attend<D, 16>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else if (nkc == 32)
    attend<D, 32>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else if (nkc == 48)
    attend<D, 48>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else
    attend<D, 64>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  st.reduce_l();

  // exact merge with the cached state, staged as bf16 rows in the q tile
  // (each warp overwrites only its own 16 rows, after its own reads of them)
  const int g = lane >> 2, t = lane & 3;
  const float log2e = 1.4426950408889634f;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = warp * 16 + g + 8 * hr;
    const float mc = m_s[r] * log2e;  // cached max, base-2 units
    const float mn = st.m[hr];
    const float M = fmaxf(mc, mn);
    const float wc = mc == neg_inf() ? 0.f : fast_exp2(mc - M);
    const float wn = mn == neg_inf() ? 0.f : fast_exp2(mn - M);
    const float L = wc * l_s[r] + wn * st.l[hr];
    const float inv = 1.f / L;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = 8 * n + 2 * t;
      const float2 oc = *reinterpret_cast<const float2*>(o_tile + (col >> 5) * 8192 +
                                                         sw128_offset(r, (col & 31) >> 2) + (col & 3) * 4);
      const float v0 = (wc * oc.x + wn * st.o[n][2 * hr]) * inv;
      const float v1 = (wc * oc.y + wn * st.o[n][2 * hr + 1]) * inv;
      *reinterpret_cast<uint32_t*>(q_tile + tile_off(r, n) + (col & 7) * 2) = pack_bf16x2(v0, v1);
    }
    const int pos = r_lo + r;
    if (a.lse != nullptr && t == 0 && pos < sm.nb && (pos < c_lo || pos >= c_hi))
      a.lse[static_cast<size_t>(sm.cus + pos) * H + h] = (M + log2f(L)) * kLn2;
  }
  __syncwarp();
  // coalesced store of this warp's 16 rows
  __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
  for (int e = lane; e < 16 * (D / 8); e += 32) {
    const int r = warp * 16 + e / (D / 8), ch = e % (D / 8);
    const int pos = r_lo + r;
    if (pos >= sm.nb || (pos >= c_lo && pos < c_hi)) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(q_tile + tile_off(r, ch));
    *reinterpret_cast<uint4*>(of + (static_cast<size_t>(sm.cus + pos) * H + h) * D + ch * 8) = v;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) step_attention_kernel(
    const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_o, const AttnArgs a, long long n_block_items, int max_pages) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full_bar[StepCfg<D>::kStages], empty_bar[StepCfg<D>::kStages], q_bar;
  __shared__ float small_a[64], small_b[64];
  __shared__ int flag;
  griddep_wait();  // q_block, the pools (and any metadata) may come from the preceding kernel
  griddep_launch_dependents();
  const long long idx = blockIdx.x;
  if (idx < n_block_items)
    block_item<D>(&tm_qb, &tm_k, &tm_v, a, smem, full_bar, empty_bar, &q_bar, small_a, small_b, &flag, idx);
  else
    merge_item<D>(&tm_q, &tm_o, a, smem, &q_bar, small_a, small_b, idx - n_block_items, max_pages);
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  PoolMaps m;
  const bool merge = plan.n_merge_items > 0;
  cudaError_t e = encode_pool_maps(a, merge, merge, &m);
  if (e != cudaSuccess) return e;
  if (!merge) m.q = m.k, m.o = m.k;  // unused by block items
  CUtensorMap tm_qb = m.k;
  if (plan.n_block_items > 0) {
    e = encode_3d_rows_sw128(&tm_qb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_block, D, a.n_heads,
                             a.bt.total_block_rows, 64, 64);
    if (e != cudaSuccess) return e;
  }
  constexpr int smem = StepCfg<D>::kSmem;
  auto kern = step_attention_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const long long grid = plan.n_block_items + plan.n_merge_items;
  const int max_pages = (a.bt.max_seq_len + kPage - 1) / kPage;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), kThreads, smem, 0, stream, tm_qb, m.k, m.v, m.q, m.o, a,
                    plan.n_block_items, max_pages);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

AttnPlan attn_plan(int batch, int n_heads, int head_dim, int max_seq_len, bool block, bool merge) {
  AttnPlan p = {};
  const int max_pages = (max_seq_len + kPage - 1) / kPage;
  // Chunks of at least two pages, at most about four chunks per (sequence, head).
  p.chunk_pages = max_pages < 1 ? 1 : (max_pages + 3) / 4;
  if (p.chunk_pages < 2) p.chunk_pages = 2;
  p.n_chunks = (max_pages + p.chunk_pages - 1) / p.chunk_pages;
  if (p.n_chunks < 1) p.n_chunks = 1;
  const long long bh = static_cast<long long>(batch) * n_heads;
  p.n_block_items = block ? bh * p.n_chunks : 0;
  p.n_merge_items = merge ? bh * max_pages : 0;
  if (block && p.n_chunks > 1) {
    p.part_bytes = align256(static_cast<size_t>(bh) * p.n_chunks * 64 * (head_dim + 4) * 4);
    p.counter_offset = p.part_bytes;
    p.total_bytes = p.counter_offset + align256(static_cast<size_t>(bh) * 4);
  }
  return p;
}

cudaError_t launch_step_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (a.bt.batch <= 0 || plan.n_block_items + plan.n_merge_items == 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, plan, stream) : launch_d<64>(a, plan, stream);
}

}  // namespace dllm
