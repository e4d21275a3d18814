// attn_stream.cu — the attention part of an inner denoising step as one
// persistent, pipelined kernel (sm_103a): the block rows' attention over
// every key of their sequence and the FACache merge of every invariant row.
//
// Work is cut into units (sequence b, head h, page p) over the real pages of
// every sequence.  The grid's CTAs (one per SM) take one of two roles, each
// walking a contiguous range of the units:
//   block role   the block queries of (b, h) (<= 64 rows, loaded once per
//                (b, h) by TMA through a 3-D tensor map over q_block) against
//                the 64 keys of page p (Fast-dLLM DualCache: [prefix KV |
//                fresh block KV | suffix KV] read through the block table).
//                The 8 compute warps split each page's keys; each keeps its
//                online-softmax state (LaCache Eq. (2)-(6)) in registers
//                across the CTA's pages of (b, h), and at the end of the
//                (b, h) the states meet in shared memory.  A (b, h) whose
//                pages span several CTAs leaves one partial state per CTA in
//                the workspace; the last CTA to arrive merges them exactly,
//                in contributor order (the same merge applied to states).
//   merge role   the rows of U in page p: the cached state (m, l, O~) merged
//                with the fresh partial state over the block keys (LaCache
//                §3.3.3, Algorithm 1 with GenStep = False).  Two groups of 4
//                warps take alternate pages.
// Half of the CTAs take the block role (a merge CTA works on two pages at a
// time, a block CTA on one), so a (b, h) spans few CTAs and its merge is
// short.  In both
// roles warp 8 streams tiles with TMA (128-byte swizzle) into an mbarrier
// ring that runs ahead across pages and (b, h) boundaries; QK^T / PV run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate), 16 query rows per warp, row
// max and sum with quad shuffles.
//
// Programmatic dependent launch: barrier setup overlaps the tail of the
// preceding kernel; every read of data it may write comes after
// griddepcontrol.wait.  Every wait is bounded; after a timeout the CTA stops
// waiting, flags DLLM_DEVERR_TIMEOUT and drains its own copies.
#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

constexpr int kThreads = 288;  // warps 0-7 compute, warp 8 streams tiles
constexpr int kMaxBatch = 512;

template <int D>
struct StreamCfg {
  static constexpr int TB = tile_bytes<D>();  // bf16 64 x D
  static constexpr int OB = 64 * D * 4;       // fp32 O~ page
  static constexpr int OS = D + 8;            // padded fp32 row of the per-warp partial states
  // block role: K/V ring | block queries | per-warp partial states
  static constexpr int kKStages = 4;
  static constexpr int KStage = 2 * TB;
  static constexpr int off_qb = kKStages * KStage;
  static constexpr int off_comb = off_qb + TB;
  static constexpr int kCombBytes = 128 * OS * 4;  // 128 (slice, row) states; later the contributors' slots
  static constexpr int kBlockSmem = off_comb + kCombBytes;
  // merge role: query page | O~ page | m | l ring, then the gathered block keys / values
  static constexpr int kMStages = 3;
  static constexpr int MStage = TB + OB + 1024;
  static constexpr int off_kc = kMStages * MStage;
  static constexpr int off_vc = off_kc + TB;
  static constexpr int kMergeSmem = off_vc + TB;
  static constexpr int kSmem = (kBlockSmem > kMergeSmem ? kBlockSmem : kMergeSmem) + 1024;  // + alignment slack
  static constexpr int PS = D + 4;  // workspace partial row: D accumulators, then (m, l)
};

struct Shared {
  uint64_t full[4], empty[4], qfull, qempty, cbar;
  int abort_flag;
  int last_flag;
  float comb_m[8 * 16], comb_l[8 * 16];  // per-warp row states of the block role
  int n_seq_units[kMaxBatch];            // H * pages of sequence b (0: invalid metadata)
  int cu[kMaxBatch + 1];                 // unit prefix
};

__device__ __forceinline__ long long split_begin(long long c, long long U, long long G) { return c * U / G; }
__device__ __forceinline__ int split_of(long long u, long long U, long long G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// Walk over the units [u, u1).
struct UWalk {
  long long u, u1;
  int b, h, p, np, first_p;
  SeqMeta sm;
  __device__ __forceinline__ void seek(const Shared& S, const BatchArgs& bt, int H) {
    int lo = 0, hi = bt.batch - 1;  // largest b with cu[b] <= u: skips sequences without units
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
      if (++h == H) seek(S, bt, H);
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

// Block-role split of a (b, h) of bb queries over the 8 compute warps:
// RG 16-row groups x KS key slices of NK = 64 / KS keys (NK a multiple of 16).
struct BlockSplit {
  int RG, KS;
  __device__ __forceinline__ explicit BlockSplit(int bb) {
    RG = (bb + 15) / 16;
    KS = RG <= 2 ? 4 : 2;
  }
  __device__ __forceinline__ bool active(int warp) const { return warp < RG * KS; }
  __device__ __forceinline__ int states() const { return KS; }  // per row group
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_stream_kernel(
    const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_o, const AttnArgs a, int n_block_ctas, int n_merge_ctas,
    int part_rows) {
  using C = StreamCfg<D>;
  constexpr int TB = C::TB, PS = C::PS, OS = C::OS, C4 = D / 4;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ Shared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  const bool block_role = static_cast<int>(blockIdx.x) < n_block_ctas;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 4; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], block_role ? 8 : 4);  // block role: all 8 warps release a page; merge: one group
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 8);
    mbar_init(&S.cbar, 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  griddep_wait();  // q_block, the pools (and any metadata) may come from the preceding kernel
  griddep_launch_dependents();
  for (int b = threadIdx.x; b < bt.batch; b += kThreads) {  // units of every sequence
    const SeqMeta m = load_meta(bt, b);
    if (!m.ok) report_error(bt.err, kErrBadShape);
    S.n_seq_units[b] = m.ok ? H * ((m.nb + kPage - 1) / kPage) : 0;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix over the sequences
    int carry = 0;
    for (int b0 = 0; b0 < bt.batch; b0 += 32) {
      const int b = b0 + lane;
      const int v = b < bt.batch ? S.n_seq_units[b] : 0;
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
  // This role's split over G = min(role CTAs, U) CTAs, so that every CTA taking
  // part owns at least one unit (the arrival count of a (b, h) assumes it).
  const long long U = S.cu[bt.batch];
  const long long n_role = block_role ? n_block_ctas : n_merge_ctas;
  const long long G = U < n_role ? U : n_role;
  const long long c = block_role ? blockIdx.x : blockIdx.x - n_block_ctas;
  if (c >= G) return;  // uniform across the CTA
  UWalk w;
  w.u = split_begin(c, U, G);
  w.u1 = split_begin(c + 1, U, G);
  w.seek(S, bt, H);

  if (block_role) {
    uint8_t* ring = smem;
    uint8_t* qb_tile = smem + C::off_qb;
    float* comb_o = reinterpret_cast<float*>(smem + C::off_comb);  // [KS * RG * 16 <= 128 (slice, row)][OS]
    if (warp == 8) {
      // ---------------------------------------------------- block producer
      if (lane == 0) {
        int nk = 0, nq = 0;
        for (; w.valid(); w.next(S, bt, H)) {
          if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
          if (w.seg_start()) {  // the block queries of (b, h)
            if (nq >= 1) wait_or_abort(S, &S.qempty, (nq - 1) & 1, bt.err);
            mbar_arrive_expect_tx(&S.qfull, TB);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              tma_load_3d(qb_tile + hf * 8192, &tm_qb, &S.qfull, hf * 64, w.h, w.sm.cub);
            ++nq;
          }
          const int s = nk % C::kKStages;
          if (nk >= C::kKStages) wait_or_abort(S, &S.empty[s], (nk / C::kKStages - 1) & 1, bt.err);
          const int y = (page_of(bt, w.b, w.p) * H + w.h) * kPage;
          uint8_t* kt = ring + s * C::KStage;
          mbar_arrive_expect_tx(&S.full[s], 2 * TB);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_2d(kt + hf * 8192, &tm_k, &S.full[s], hf * 64, y);
            tma_load_2d(kt + TB + hf * 8192, &tm_v, &S.full[s], hf * 64, y);
          }
          ++nk;
        }
        for (int i = (nk > C::kKStages ? nk - C::kKStages : 0); i < nk; ++i)  // every copy has landed
          if (!mbar_wait(&S.full[i % C::kKStages], (i / C::kKStages) & 1)) report_error(bt.err, kErrTimeout);
        if (nq >= 1 && !mbar_wait(&S.qfull, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
      }
      return;
    }
    // ------------------------------------------------ block compute (warps 0-7)
    const int g = lane >> 2, t = lane & 3;
    int nk = 0, nq = 0, ncb = 0;  // K/V pages, query tiles, combine passes so far
    WarpAttn<D> st;
    uint32_t qf[D / 16][4];
    __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
    for (; w.valid(); w.next(S, bt, H)) {
      const BlockSplit sp(w.sm.bb);
      const bool active = sp.active(warp);
      const int rg = warp % sp.RG, ks = warp / sp.RG;
      if (w.seg_start()) {
        wait_or_abort(S, &S.qfull, nq & 1, bt.err);
        if (active) load_q_frags<D>(qf, smem_u32(qb_tile), rg * 16, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.qempty);
        ++nq;
        st.init();
      }
      const int s = nk % C::kKStages;
      wait_or_abort(S, &S.full[s], (nk / C::kKStages) & 1, bt.err);
      if (active) {
        const uint32_t kt = smem_u32(ring + s * C::KStage), vt = kt + TB;
        const int base = w.p * kPage, nb = w.sm.nb;
        auto valid = [base, nb](int key) { return base + key < nb; };
        if (sp.KS == 4)
          attend<D, 16>(st, qf, kt, vt, ks * 16, a.scale_log2, valid, lane);
        else
          attend<D, 32>(st, qf, kt, vt, ks * 32, a.scale_log2, valid, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
      ++nk;
      if (!w.seg_end()) continue;

      // ---- (b, h) segment complete on this CTA: combine the KS states of each row in shared memory
      if (active) {
        st.reduce_l();
        const int slot0 = ks * sp.RG * 16 + rg * 16 + g, slot1 = slot0 + 8;
        if (t == 0) {
          S.comb_m[slot0] = st.m[0];
          S.comb_l[slot0] = st.l[0];
          S.comb_m[slot1] = st.m[1];
          S.comb_l[slot1] = st.l[1];
        }
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          *reinterpret_cast<float2*>(comb_o + slot0 * OS + 8 * n + 2 * t) = make_float2(st.o[n][0], st.o[n][1]);
          *reinterpret_cast<float2*>(comb_o + slot1 * OS + 8 * n + 2 * t) = make_float2(st.o[n][2], st.o[n][3]);
        }
      }
      named_barrier(1, 256);
      const size_t row0 = static_cast<size_t>(w.sm.cus + w.sm.sb) * H + w.h;  // o_full / lse row of block row 0
      const bool whole = w.seg_whole();
      const long long s_bh = S.cu[w.b] + static_cast<long long>(w.h) * w.np, e_bh = s_bh + w.np;
      const int my_slot = (split_begin(c, U, G) >= s_bh) ? 0 : 1;  // first / last segment of this CTA
      float* mine = a.part + ((static_cast<size_t>(c) * 2 + my_slot) * part_rows) * PS;
      for (int item = threadIdx.x; item < w.sm.bb * C4; item += 256) {
        const int i = item / C4, col = (item % C4) * 4;
        float M = neg_inf();
        for (int q = 0; q < sp.states(); ++q) M = fmaxf(M, S.comb_m[q * sp.RG * 16 + i]);
        const float Mu = M == neg_inf() ? 0.f : M;
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < sp.states(); ++q) {
          const int slot = q * sp.RG * 16 + i;
          const float wgt = fast_exp2(S.comb_m[slot] - Mu);
          L += wgt * S.comb_l[slot];
          const float4 ov = *reinterpret_cast<const float4*>(comb_o + slot * OS + col);
          acc.x += wgt * ov.x;
          acc.y += wgt * ov.y;
          acc.z += wgt * ov.z;
          acc.w += wgt * ov.w;
        }
        if (whole) {  // every page of (b, h) was here: finish the row
          const float inv = 1.f / L;
          const size_t orow = row0 + static_cast<size_t>(i) * H;
          uint2 pk;
          pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
          *reinterpret_cast<uint2*>(of + orow * D + col) = pk;
          if (a.lse != nullptr && col == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
        } else {
          *reinterpret_cast<float4*>(mine + i * PS + col) = acc;
          if (col == 0) *reinterpret_cast<float2*>(mine + i * PS + D) = make_float2(M, L);
        }
      }
      named_barrier(1, 256);  // comb is free again; the partial rows are written ...
      if (whole) continue;
      const int c_first = split_of(s_bh, U, G), c_last = split_of(e_bh - 1, U, G);
      int32_t* counter = a.counters + static_cast<size_t>(w.b) * H + w.h;
      if (threadIdx.x == 0) {
        __threadfence();  // ... and (cumulatively) visible GPU-wide before the arrival is counted
        S.last_flag = atomicAdd(counter, 1) == c_last - c_first;
      }
      named_barrier(1, 256);
      if (!S.last_flag) continue;
      __threadfence();
      // Last arrival: merge every contributor's state (this CTA's too, as
      // written) in contributor order, so the rounding does not depend on
      // which CTA arrives last.  The contributors' slots come into the idle
      // key-slice buffer with bulk copies, as many at once as fit, so each
      // pass costs one round trip however many rows and contributors it has.
      const int n_contrib = c_last - c_first + 1;
      const float* slot_first =
          a.part + (static_cast<size_t>(c_first) * 2 + (split_begin(c_first, U, G) < s_bh ? 1 : 0)) * part_rows * PS;
      const size_t cta_stride = static_cast<size_t>(2) * part_rows * PS;
      auto slot_of = [&](int k) { return k == 0 ? slot_first : a.part + static_cast<size_t>(c_first + k) * cta_stride; };
      const uint32_t slot_bytes = static_cast<uint32_t>(w.sm.bb) * PS * 4;
      const int fit = C::kCombBytes / static_cast<int>(slot_bytes);  // slots the buffer holds (>= 2)
      // one pass if every contributor fits; otherwise the last slot keeps the running state
      const int per_pass = n_contrib <= fit ? fit : fit - 1;
      float* stage = comb_o;  // [fit][bb][PS]
      // Passes of per_pass contributors (one pass in all but the largest
      // splits); between passes the running (max, sum, accumulators) of each
      // row wait in the buffer's last slot.
      float* keep = stage + static_cast<size_t>(fit - 1) * w.sm.bb * PS;
      for (int k0 = 0; k0 < n_contrib; k0 += per_pass) {
        const int nk = min(per_pass, n_contrib - k0);
        const bool first = k0 == 0, last_pass = k0 + nk >= n_contrib;
        if (threadIdx.x == 0) {
          // order the other contributors' writes (acquired above) and this CTA's earlier generic
          // accesses of the buffer before the async-proxy copies
          asm volatile("fence.proxy.async;" ::: "memory");
          mbar_arrive_expect_tx(&S.cbar, slot_bytes * nk);
          for (int k = 0; k < nk; ++k) bulk_load(stage + k * w.sm.bb * PS, slot_of(k0 + k), slot_bytes, &S.cbar);
        }
        wait_or_abort(S, &S.cbar, ncb & 1, bt.err);
        ++ncb;
        for (int item = threadIdx.x; item < w.sm.bb * C4; item += 256) {
          const int i = item / C4, col = (item % C4) * 4;
          float* kr = keep + i * PS;
          float Mprev = neg_inf(), Lprev = 0.f;
          float4 Aprev = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!first) {
            Aprev = *reinterpret_cast<const float4*>(kr + col);
            const float2 ml = *reinterpret_cast<const float2*>(kr + D);  // the row's, from the previous pass
            Mprev = ml.x;
            Lprev = ml.y;
          }
          float M = Mprev;
          for (int k = 0; k < nk; ++k) M = fmaxf(M, stage[(k * w.sm.bb + i) * PS + D]);
          const float Mu = M == neg_inf() ? 0.f : M;
          const float r = fast_exp2(Mprev - Mu);  // rescales the earlier passes (0 before the first)
          float L = r * Lprev;
          float4 acc = make_float4(r * Aprev.x, r * Aprev.y, r * Aprev.z, r * Aprev.w);
          for (int k = 0; k < nk; ++k) {
            const float* pr = stage + (k * w.sm.bb + i) * PS;
            const float wgt = fast_exp2(pr[D] - Mu);
            L += wgt * pr[D + 1];
            const float4 ov = *reinterpret_cast<const float4*>(pr + col);
            acc.x += wgt * ov.x;
            acc.y += wgt * ov.y;
            acc.z += wgt * ov.z;
            acc.w += wgt * ov.w;
          }
          if (last_pass) {
            const float inv = 1.f / L;
            const size_t orow = row0 + static_cast<size_t>(i) * H;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(of + orow * D + col) = pk;
            if (a.lse != nullptr && col == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
          } else {
            // every item of a row computes the same (M, L); the column-0 item keeps it for the
            // next pass (read there by the row's other items, after the barrier below)
            *reinterpret_cast<float4*>(kr + col) = acc;
            if (col == 0) *reinterpret_cast<float2*>(kr + D) = make_float2(M, L);
          }
        }
        named_barrier(1, 256);  // the staged slots are consumed before the next pass overwrites them
      }
      if (threadIdx.x == 0) *counter = 0;  // ready for the next call
      named_barrier(1, 256);  // comb_m is reused by the next segment
    }
    return;
  }

  // ===================================================================== merge role
  uint8_t* ring = smem;
  uint8_t* kc_tile = smem + C::off_kc;
  uint8_t* vc_tile = smem + C::off_vc;
  if (warp == 8) {
    // ---------------------------------------------------- merge producer
    if (lane == 0) {
      int nm = 0;
      for (; w.valid(); w.next(S, bt, H)) {
        if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
        if (!w.has_u_rows()) continue;
        const int s = nm % C::kMStages;
        if (nm >= C::kMStages) wait_or_abort(S, &S.empty[s], (nm / C::kMStages - 1) & 1, bt.err);
        const int y = (page_of(bt, w.b, w.p) * H + w.h) * kPage;
        uint8_t* mt = ring + s * C::MStage;
        mbar_arrive_expect_tx(&S.full[s], TB + C::OB + 512);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(mt + hf * 8192, &tm_q, &S.full[s], hf * 64, y);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) tma_load_2d(mt + TB + j * 8192, &tm_o, &S.full[s], j * 32, y);
        bulk_load(mt + TB + C::OB, a.m_pool + y, 256, &S.full[s]);
        bulk_load(mt + TB + C::OB + 256, a.l_pool + y, 256, &S.full[s]);
        ++nm;
      }
      for (int i = (nm > C::kMStages ? nm - C::kMStages : 0); i < nm; ++i)  // every copy has landed
        if (!mbar_wait(&S.full[i % C::kMStages], (i / C::kMStages) & 1)) report_error(bt.err, kErrTimeout);
    }
    return;
  }
  // ------------------------------------------------ merge compute (2 groups of 4 warps)
  const int grp = warp >> 2, mw = warp & 3;
  const int g = lane >> 2, t = lane & 3;
  const float log2e = 1.4426950408889634f;
  int nm = 0;  // pages with U rows seen so far (both groups count all of them)
  int nkc = 32;
  __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
  for (; w.valid(); w.next(S, bt, H)) {
    if (w.seg_start()) {  // gather the fresh block keys / values of (b, h) through the table
      named_barrier(2, 256);  // both groups are done with the previous (b, h)'s
      nkc = w.sm.bb <= 32 ? 32 : 64;  // keys the QK^T below covers; rows past bb are zero
      const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
      const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
      for (int e = threadIdx.x; e < nkc * (D / 8); e += 256) {
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
      named_barrier(2, 256);
    }
    if (!w.has_u_rows()) continue;
    const int mine = (nm & 1) == grp;
    const int s = nm % C::kMStages;
    const int uses = nm / C::kMStages;
    ++nm;
    if (!mine) continue;  // the other group's page
    wait_or_abort(S, &S.full[s], uses & 1, bt.err);
    uint8_t* q_tile = ring + s * C::MStage;
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
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  PoolMaps m;
  const bool merge = plan.n_merge_ctas > 0, block = plan.n_block_ctas > 0;
  cudaError_t e = encode_pool_maps(a, merge, merge, &m);
  if (e != cudaSuccess) return e;
  if (!merge) m.q = m.k, m.o = m.k;  // unused without the merge role
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
  return launch_pdl(kern, dim3(plan.n_block_ctas + plan.n_merge_ctas), kThreads, smem, 0, stream, tm_qb, m.k, m.v,
                    m.q, m.o, a, plan.n_block_ctas, plan.n_merge_ctas, plan.part_rows);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

AttnPlan attn_plan(int batch, int n_heads, int head_dim, int max_seq_len, int max_block_len, int num_sms, bool block,
                   bool merge) {
  AttnPlan p = {};
  const long long max_pages = (max_seq_len + kPage - 1) / kPage;
  const long long units = static_cast<long long>(batch) * n_heads * max_pages;  // upper bound of either role's units
  const int g = static_cast<int>(units < num_sms ? (units < 1 ? 1 : units) : num_sms);
  p.part_rows = max_block_len < 1 ? 1 : max_block_len;
  if (block && merge) {
    // one block-role CTA per (b, h) (so that no (b, h) needs a cross-CTA merge)
    // while that is at most half of the CTAs; the rest take the merge role
    const long long bh = static_cast<long long>(batch) * n_heads;
    const int half = g / 2 < 1 ? 1 : g / 2;
    p.n_block_ctas = bh < half ? static_cast<int>(bh) : half;
    p.n_merge_ctas = g - p.n_block_ctas < 1 ? 1 : g - p.n_block_ctas;
  } else {
    p.n_block_ctas = block ? g : 0;
    p.n_merge_ctas = merge ? g : 0;
  }
  if (block) {  // two partial slots per block CTA (its first and last (b, h)) and one counter per (b, h)
    p.part_bytes = align256(static_cast<size_t>(p.n_block_ctas) * 2 * p.part_rows * (head_dim + 4) * 4);
    p.counter_offset = p.part_bytes;
    p.total_bytes = p.counter_offset + align256(static_cast<size_t>(batch) * n_heads * 4);
  }
  return p;
}

bool attn_batch_supported(int batch) { return batch <= kMaxBatch; }

cudaError_t launch_step_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (a.bt.batch <= 0 || plan.n_block_ctas + plan.n_merge_ctas == 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, plan, stream) : launch_d<64>(a, plan, stream);
}

}  // namespace dllm
