// attn_stream.cu — the attention part of an inner denoising step as one
// persistent, pipelined kernel (sm_103a): the block rows' attention over
// every key of their sequence and the FACache merge of every invariant row.
//
// Work is cut into units (sequence b, head h, page p) over the real pages of
// every sequence; CTA c (one per SM) owns the contiguous unit range
// [c U / G, (c + 1) U / G), so it walks consecutive pages of one (b, h) at a
// time.  For each unit:
//   block part   the block queries of (b, h) (<= 64 rows, loaded once per
//                (b, h) by TMA through a 3-D tensor map over q_block) against
//                the 64 keys of page p (Fast-dLLM DualCache: [prefix KV |
//                fresh block KV | suffix KV] read through the block table);
//                the online-softmax state (LaCache Eq. (2)-(6)) runs on in
//                registers across the CTA's pages of (b, h).  A (b, h) whose
//                pages span several CTAs leaves one partial state per CTA in
//                the workspace and the last of them to arrive merges them
//                exactly (the same merge applied to states).
//   merge part   the rows of U in page p: the cached state (m, l, O~) merged
//                with the fresh partial state over the block keys (LaCache
//                §3.3.3, Algorithm 1 with GenStep = False).
// Warps 0-3 run the block part, warps 4-7 the merge part, warp 8 streams
// tiles with TMA into two mbarrier rings (K/V pages; query page + fp32 O~
// page + m, l), running ahead across units and (b, h) boundaries, so a CTA
// keeps ~160 KB of loads in flight instead of paying a load latency per
// short-lived CTA.  QK^T / PV run on mma.sync m16n8k16 (bf16 in, fp32
// accumulate), 16 query rows per warp; row max and sum use quad shuffles.
//
// Programmatic dependent launch: barrier setup overlaps the tail of the
// preceding kernel; every read of data it may write comes after
// griddepcontrol.wait.  Every wait is bounded; after a timeout the CTA stops
// waiting, flags DLLM_DEVERR_TIMEOUT and drains its own copies.
#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

constexpr int kThreads = 288;  // warps 0-3 block part, 4-7 merge part, 8 producer
constexpr int kMaxBatch = 512;

template <int D>
struct StreamCfg {
  static constexpr int TB = tile_bytes<D>();   // bf16 64 x D
  static constexpr int OB = 64 * D * 4;        // fp32 O~ page
  static constexpr int KStage = 2 * TB;        // K page | V page
  static constexpr int MStage = TB + OB + 1024;  // q page | O~ page | m (256 B) | l (256 B), padded
  static constexpr int kKStages = 2, kMStages = 2;
  static constexpr int off_m = kKStages * KStage;
  static constexpr int off_qb = off_m + kMStages * MStage;
  static constexpr int off_kc = off_qb + TB;
  static constexpr int off_vc = off_kc + TB;
  static constexpr int kSmem = off_vc + TB + 1024;  // + alignment slack
  static constexpr int PS = D + 4;                  // workspace partial row: D accumulators, then (m, l)
};

struct Shared {
  uint64_t kfull[2], kempty[2], mfull[2], mempty[2], qfull, qempty;
  int abort_flag;
  int last_flag;
  int n_seq_units[kMaxBatch];  // H * pages of sequence b (0: invalid metadata)
  int cu[kMaxBatch + 1];       // unit prefix
};

__device__ __forceinline__ long long cta_begin(long long c, long long U, long long G) { return c * U / G; }
__device__ __forceinline__ int cta_of(long long u, long long U, long long G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// Walk over the real units [u, u1) of this CTA.
struct UWalk {
  long long u, u1;
  int b, h, p, np, first_p;
  SeqMeta sm;
  __device__ __forceinline__ void seek(const Shared& S, const BatchArgs& bt, int H) {
    int lo = 0, hi = bt.batch - 1;  // largest b with cu[b] <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (S.cu[mid] <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    b = lo;
    np = S.n_seq_units[b] / H;
    const int r = static_cast<int>(u - S.cu[b]);
    h = r / np;
    p = r % np;
    first_p = p;
    sm = load_meta(bt, b);
  }
  __device__ __forceinline__ bool valid() const { return u < u1; }
  __device__ __forceinline__ bool seg_start() const { return p == first_p; }
  __device__ __forceinline__ bool seg_end() const { return u + 1 == u1 || p == np - 1; }
  __device__ __forceinline__ bool seg_whole() const { return first_p == 0 && p == np - 1; }
  __device__ __forceinline__ bool has_u_rows() const {
    const int r_lo = p * kPage, r_hi = min(sm.nb, r_lo + kPage);
    return r_lo < sm.sb || r_hi > sm.sb + sm.bb;
  }
  __device__ __forceinline__ void next(const Shared& S, const BatchArgs& bt, int H) {
    ++u;
    if (u >= u1) return;
    if (++p == np) {
      p = 0;
      if (++h == H) seek(S, bt, H);  // next sequence with units (p = 0 there)
      first_p = 0;
    }
  }
};

// Bounded wait that gives up (and makes the whole CTA give up) after a timeout.
__device__ __forceinline__ void wait_or_abort(Shared& S, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return;
  if (!mbar_wait(bar, parity)) {
    S.abort_flag = 1;
    report_error(err, kErrTimeout);
  }
}

template <int D>
__device__ __forceinline__ void store_row_pair(__nv_bfloat16* of, size_t orow, const float (&o)[D / 8][4], int hr,
                                               float inv, int t) {
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
    *reinterpret_cast<uint32_t*>(of + orow * D + 8 * n + 2 * t) =
        pack_bf16x2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_stream_kernel(
    const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_o, const AttnArgs a, int do_block, int do_merge, int part_rows) {
  using C = StreamCfg<D>;
  constexpr int TB = C::TB, PS = C::PS, C4 = D / 4;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ Shared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.kfull[s], 1);
      mbar_init(&S.kempty[s], 4);
      mbar_init(&S.mfull[s], 1);
      mbar_init(&S.mempty[s], 4);
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 4);
    S.abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  griddep_wait();  // q_block, the pools (and any metadata) may come from the preceding kernel
  griddep_launch_dependents();
  // units of every sequence (metadata that contradicts the host bounds: none)
  for (int b = threadIdx.x; b < bt.batch; b += kThreads) {
    const SeqMeta m = load_meta(bt, b);
    if (!m.ok) report_error(bt.err, kErrBadShape);
    S.n_seq_units[b] = m.ok ? H * ((m.nb + kPage - 1) / kPage) : 0;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over the sequences
    int carry = 0;
    for (int b0 = 0; b0 < bt.batch; b0 += 32) {
      const int b = b0 + lane;
      int v = b < bt.batch ? S.n_seq_units[b] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (b < bt.batch) S.cu[b] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) S.cu[bt.batch] = carry;
  }
  __syncthreads();
  // Split over G = min(grid, U) CTAs so that every CTA taking part owns at
  // least one unit (the arrival count of a (b, h) assumes it).
  const long long U = S.cu[bt.batch];
  const long long G = U < static_cast<long long>(gridDim.x) ? U : static_cast<long long>(gridDim.x);
  if (static_cast<long long>(blockIdx.x) >= G) return;  // uniform across the CTA
  UWalk w;
  w.u = cta_begin(blockIdx.x, U, G);
  w.u1 = cta_begin(blockIdx.x + 1, U, G);
  if (w.u >= w.u1) return;  // no units (uniform across the CTA)
  w.seek(S, bt, H);
  uint8_t* ring_k = smem;
  uint8_t* ring_m = smem + C::off_m;
  uint8_t* qb_tile = smem + C::off_qb;
  uint8_t* kc_tile = smem + C::off_kc;
  uint8_t* vc_tile = smem + C::off_vc;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int nk = 0, nm = 0, nq = 0;
      for (; w.valid(); w.next(S, bt, H)) {
        if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
        const int pg = page_of(bt, w.b, w.p);
        const int y = (pg * H + w.h) * kPage;
        if (do_block) {
          if (w.seg_start()) {  // the block queries of (b, h)
            if (nq >= 1) wait_or_abort(S, &S.qempty, (nq - 1) & 1, bt.err);
            mbar_arrive_expect_tx(&S.qfull, TB);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              tma_load_3d(qb_tile + hf * 8192, &tm_qb, &S.qfull, hf * 64, w.h, w.sm.cub);
            ++nq;
          }
          const int s = nk & 1;
          if (nk >= 2) wait_or_abort(S, &S.kempty[s], ((nk >> 1) - 1) & 1, bt.err);
          uint8_t* kt = ring_k + s * C::KStage;
          mbar_arrive_expect_tx(&S.kfull[s], 2 * TB);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_2d(kt + hf * 8192, &tm_k, &S.kfull[s], hf * 64, y);
            tma_load_2d(kt + TB + hf * 8192, &tm_v, &S.kfull[s], hf * 64, y);
          }
          ++nk;
        }
        if (do_merge && w.has_u_rows()) {
          const int s = nm & 1;
          if (nm >= 2) wait_or_abort(S, &S.mempty[s], ((nm >> 1) - 1) & 1, bt.err);
          uint8_t* mt = ring_m + s * C::MStage;
          mbar_arrive_expect_tx(&S.mfull[s], TB + C::OB + 512);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(mt + hf * 8192, &tm_q, &S.mfull[s], hf * 64, y);
#pragma unroll
          for (int j = 0; j < D / 32; ++j) tma_load_2d(mt + TB + j * 8192, &tm_o, &S.mfull[s], j * 32, y);
          bulk_load(mt + TB + C::OB, a.m_pool + y, 256, &S.mfull[s]);
          bulk_load(mt + TB + C::OB + 256, a.l_pool + y, 256, &S.mfull[s]);
          ++nm;
        }
      }
      // every issued copy has landed before the CTA can exit
      for (int i = (nk > 2 ? nk - 2 : 0); i < nk; ++i)
        if (!mbar_wait(&S.kfull[i & 1], (i >> 1) & 1)) report_error(bt.err, kErrTimeout);
      for (int i = (nm > 2 ? nm - 2 : 0); i < nm; ++i)
        if (!mbar_wait(&S.mfull[i & 1], (i >> 1) & 1)) report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.qfull, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
    }
  } else if (warp < 4) {
    // ------------------------------------------------ block part (warps 0-3)
    if (!do_block) return;
    const int g = lane >> 2, t = lane & 3;
    int nk = 0, nq = 0;
    WarpAttn<D> st;
    uint32_t qf[D / 16][4];
    __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
    for (; w.valid(); w.next(S, bt, H)) {
      const int RG = (w.sm.bb + 15) / 16;
      const bool active = warp < RG;
      if (w.seg_start()) {
        wait_or_abort(S, &S.qfull, nq & 1, bt.err);
        if (active) load_q_frags<D>(qf, smem_u32(qb_tile), warp * 16, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.qempty);
        ++nq;
        st.init();
      }
      const int s = nk & 1;
      wait_or_abort(S, &S.kfull[s], (nk >> 1) & 1, bt.err);
      if (active) {
        const uint32_t kt = smem_u32(ring_k + s * C::KStage), vt = kt + TB;
        const int base = w.p * kPage, nb = w.sm.nb;
        attend<D, 64>(st, qf, kt, vt, 0, a.scale_log2, [base, nb](int key) { return base + key < nb; }, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.kempty[s]);
      ++nk;
      if (!w.seg_end()) continue;

      // ---- (b, h) segment complete on this CTA
      if (active) st.reduce_l();
      const size_t row0 = static_cast<size_t>(w.sm.cus + w.sm.sb) * H + w.h;  // o_full / lse row of block row 0
      if (w.seg_whole()) {  // every page of (b, h) was here: finish the rows
        if (active) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int i = warp * 16 + g + 8 * hr;
            if (i >= w.sm.bb) continue;
            const size_t orow = row0 + static_cast<size_t>(i) * H;
            store_row_pair<D>(of, orow, st.o, hr, 1.f / st.l[hr], t);
            if (a.lse != nullptr && t == 0) a.lse[orow] = (st.m[hr] + log2f(st.l[hr])) * kLn2;
          }
        }
        continue;
      }
      // partial state of this CTA's pages of (b, h) -> workspace slot (CTA, first/last segment)
      const long long s_bh = S.cu[w.b] + static_cast<long long>(w.h) * w.np, e_bh = s_bh + w.np;
      const int my_slot = (cta_begin(blockIdx.x, U, G) >= s_bh) ? 0 : 1;
      if (active) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = warp * 16 + g + 8 * hr;
          if (i >= w.sm.bb) continue;
          float* pr = a.part + ((static_cast<size_t>(blockIdx.x) * 2 + my_slot) * part_rows + i) * PS;
#pragma unroll
          for (int n = 0; n < D / 8; ++n)
            *reinterpret_cast<float2*>(pr + 8 * n + 2 * t) = make_float2(st.o[n][2 * hr], st.o[n][2 * hr + 1]);
          if (t == 0) *reinterpret_cast<float2*>(pr + D) = make_float2(st.m[hr], st.l[hr]);
        }
      }
      const int c_first = cta_of(s_bh, U, G), c_last = cta_of(e_bh - 1, U, G);
      int32_t* counter = a.counters + static_cast<size_t>(w.b) * H + w.h;
      named_barrier(1, 128);  // the partial rows are written ...
      if (threadIdx.x == 0) {
        __threadfence();  // ... and (cumulatively) visible GPU-wide before the arrival is counted
        S.last_flag = atomicAdd(counter, 1) == c_last - c_first;
      }
      named_barrier(1, 128);
      if (!S.last_flag) continue;
      __threadfence();
      // Last arrival: merge every contributor's state (this CTA's own too, as
      // written) in contributor order, so the rounding does not depend on
      // which CTA arrives last.  Fragment layout: every thread reads exactly
      // the (row, column) pairs it holds, one contributor's loads issued
      // together.
      if (active) {
        const float* slot0 =
            a.part + (static_cast<size_t>(c_first) * 2 + (cta_begin(c_first, U, G) < s_bh ? 1 : 0)) * part_rows * PS;
        const size_t cta_stride = static_cast<size_t>(2) * part_rows * PS;
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int i = warp * 16 + g + 8 * hr;
          if (i >= w.sm.bb) continue;
          float M = neg_inf();
          for (int c = c_first; c <= c_last; ++c) {
            const float* pr = (c == c_first ? slot0 : a.part + static_cast<size_t>(c) * cta_stride) + i * PS;
            M = fmaxf(M, __ldcg(pr + D));
          }
          const float Mu = M == neg_inf() ? 0.f : M;
          float L = 0.f;
#pragma unroll
          for (int n = 0; n < D / 8; ++n) st.o[n][2 * hr] = st.o[n][2 * hr + 1] = 0.f;
          for (int c = c_first; c <= c_last; ++c) {
            const float* pr = (c == c_first ? slot0 : a.part + static_cast<size_t>(c) * cta_stride) + i * PS;
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(pr + D));
            float2 v[D / 8];
#pragma unroll
            for (int n = 0; n < D / 8; ++n) v[n] = __ldcg(reinterpret_cast<const float2*>(pr + 8 * n + 2 * t));
            const float wc = fast_exp2(ml.x - Mu);
            L += wc * ml.y;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
              st.o[n][2 * hr] += wc * v[n].x;
              st.o[n][2 * hr + 1] += wc * v[n].y;
            }
          }
          const size_t orow = row0 + static_cast<size_t>(i) * H;
          store_row_pair<D>(of, orow, st.o, hr, 1.f / L, t);
          if (a.lse != nullptr && t == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
        }
      }
      if (threadIdx.x == 0) *counter = 0;  // ready for the next call
    }
  } else {
    // ------------------------------------------------ merge part (warps 4-7)
    if (!do_merge) return;
    const int mw = warp - 4, mt_id = threadIdx.x - 128;  // merge warp, thread among the 128
    const int g = lane >> 2, t = lane & 3;
    const float log2e = 1.4426950408889634f;
    int nm = 0;
    int nkc = 32;
    __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
    for (; w.valid(); w.next(S, bt, H)) {
      if (w.seg_start()) {  // gather the fresh block keys / values of (b, h) through the table
        named_barrier(2, 128);  // the previous (b, h)'s readers are done with them
        nkc = w.sm.bb <= 32 ? 32 : 64;  // keys the QK^T below covers; rows past bb are zero
        const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
        const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
        for (int e = mt_id; e < nkc * (D / 8); e += 128) {
          const int cc = e / (D / 8), ch = e % (D / 8);
          uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
          if (cc < w.sm.bb) {
            const int pos = w.sm.sb + cc;
            const int pgc = page_of(bt, w.b, pos / kPage);
            const size_t off = ((static_cast<size_t>(pgc) * H + w.h) * kPage + (pos % kPage)) * D;
            kv4 = __ldg(reinterpret_cast<const uint4*>(kp + off) + ch);
            vv4 = __ldg(reinterpret_cast<const uint4*>(vp + off) + ch);
          }
          *reinterpret_cast<uint4*>(kc_tile + tile_off(cc, ch)) = kv4;
          *reinterpret_cast<uint4*>(vc_tile + tile_off(cc, ch)) = vv4;
        }
        named_barrier(2, 128);
      }
      if (!w.has_u_rows()) continue;
      const int s = nm & 1;
      wait_or_abort(S, &S.mfull[s], (nm >> 1) & 1, bt.err);
      uint8_t* q_tile = ring_m + s * C::MStage;
      const uint8_t* o_tile = q_tile + TB;
      const float* m_s = reinterpret_cast<const float*>(q_tile + TB + C::OB);
      const float* l_s = m_s + 64;
      // fresh partial state over the block keys (Eq. (2)-(6) from the empty state)
      WarpAttn<D> st;
      st.init();
      uint32_t qf[D / 16][4];
      load_q_frags<D>(qf, smem_u32(q_tile), mw * 16, lane);
      const uint32_t kt = smem_u32(kc_tile), vt = smem_u32(vc_tile);
      const int bb = w.sm.bb;
      auto valid = [bb](int key) { return key < bb; };
      if (nkc <= 32)
        attend<D, 32>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
      else
        attend<D, 64>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
      st.reduce_l();
      // exact merge with the cached state, staged as bf16 rows in this warp's
      // 16 rows of the q tile (read into registers above)
      const int r_lo = w.p * kPage, c_lo = w.sm.sb, c_hi = w.sm.sb + w.sm.bb;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = mw * 16 + g + 8 * hr;
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
        if (a.lse != nullptr && t == 0 && pos < w.sm.nb && (pos < c_lo || pos >= c_hi))
          a.lse[static_cast<size_t>(w.sm.cus + pos) * H + w.h] = (M + log2f(L)) * kLn2;
      }
      __syncwarp();
      for (int e = lane; e < 16 * (D / 8); e += 32) {  // coalesced store of this warp's 16 rows
        const int r = mw * 16 + e / (D / 8), ch = e % (D / 8);
        const int pos = r_lo + r;
        if (pos >= w.sm.nb || (pos >= c_lo && pos < c_hi)) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(q_tile + tile_off(r, ch));
        *reinterpret_cast<uint4*>(of + (static_cast<size_t>(w.sm.cus + pos) * H + w.h) * D + ch * 8) = v;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.mempty[s]);
      ++nm;
    }
  }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  PoolMaps m;
  const bool merge = plan.n_merge_items > 0, block = plan.n_block_items > 0;
  cudaError_t e = encode_pool_maps(a, merge, merge, &m);
  if (e != cudaSuccess) return e;
  if (!merge) m.q = m.k, m.o = m.k;  // unused without the merge part
  CUtensorMap tm_qb = m.k;
  if (block) {
    e = encode_3d_rows_sw128(&tm_qb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_block, D, a.n_heads,
                             a.bt.total_block_rows, 64, 64);
    if (e != cudaSuccess) return e;
  }
  constexpr int smem = StreamCfg<D>::kSmem;
  auto kern = attn_stream_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(plan.grid), kThreads, smem, 0, stream, tm_qb, m.k, m.v, m.q, m.o, a,
                    block ? 1 : 0, merge ? 1 : 0, plan.part_rows);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

AttnPlan attn_plan(int batch, int n_heads, int head_dim, int max_seq_len, int max_block_len, int num_sms, bool block,
                   bool merge) {
  AttnPlan p = {};
  const long long max_pages = (max_seq_len + kPage - 1) / kPage;
  const long long units = static_cast<long long>(batch) * n_heads * max_pages;  // upper bound
  p.grid = static_cast<int>(units < num_sms ? (units < 1 ? 1 : units) : num_sms);
  p.part_rows = max_block_len < 1 ? 1 : max_block_len;
  p.n_block_items = block ? units : 0;
  p.n_merge_items = merge ? units : 0;
  if (block) {  // two partial slots per CTA (its first and last (b, h) segments) and one counter per (b, h)
    p.part_bytes = align256(static_cast<size_t>(p.grid) * 2 * p.part_rows * (head_dim + 4) * 4);
    p.counter_offset = p.part_bytes;
    p.total_bytes = p.counter_offset + align256(static_cast<size_t>(batch) * n_heads * 4);
  }
  return p;
}

bool attn_batch_supported(int batch) { return batch <= kMaxBatch; }

cudaError_t launch_step_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (a.bt.batch <= 0 || plan.n_block_items + plan.n_merge_items == 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, plan, stream) : launch_d<64>(a, plan, stream);
}

}  // namespace dllm
