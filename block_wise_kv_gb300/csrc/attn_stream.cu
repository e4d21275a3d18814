// attn_stream.cu — the attention part of an inner denoising step as one
// persistent, pipelined kernel (sm_103a): the block rows' attention over
// every key of their sequence and the FACache merge of every invariant row.
//
// The grid's CTAs (one per SM) take one of two roles:
//   block role   a contiguous range of (sequence b, head h) pairs, each owned
//                whole by one CTA: the block queries (<= 64 rows) against all
//                of the sequence's pages (Fast-dLLM DualCache: [prefix KV |
//                fresh block KV | suffix KV] read through the block table),
//                S = Q K^T and O += P V on the 5th-generation tensor cores
//                with the accumulators in tensor memory, online softmax
//                (LaCache Eq. (2)-(6)) between the two MMAs.  No state leaves
//                the CTA before O / l is final.
//   merge role   a contiguous range of units (b, h, page p) over the real
//                pages of every sequence: the rows of U in page p, the cached
//                state (m, l, O~) merged with the fresh partial state over
//                the block keys (LaCache §3.3.3, Algorithm 1 with GenStep =
//                False), on mma.sync m16n8k16 (bf16 in, fp32 accumulate); three
//                groups of 4 warps take the pages in turn.  The cached O~ is
//                stored as O~ / l in fp16.
// The host splits the CTAs between the roles by their work (attn_plan); a
// (b, h) pair is never split between block-role CTAs.  The tiles are streamed
// with TMA (128-byte swizzle) into mbarrier rings that run ahead across pages
// and (b, h) boundaries: by a producer warp in the block role, by the leader
// of the consuming group (refilling the stage it just freed) in the merge role.
//
// Programmatic dependent launch: barrier setup, the metadata prefix and the
// loads of data the preceding kernel does not write (pages without block
// rows) overlap that kernel's tail; every read of data it may write comes
// after griddepcontrol.wait.  Every wait is bounded; after a timeout the CTA
// stops waiting, flags DLLM_DEVERR_TIMEOUT and drains its own copies.
#include <math.h>

#include <algorithm>

#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

constexpr int kThreads = 384;
// Time of a merge-role page over that of a block-role page on GB300, for blocks of at most
// 32 rows and for longer ones (the block role packs four 32-row query sets or two 64-row
// ones into a tile; the merge attends to 32 or 64 keys), fitted to sweeps of the split:
// 32-layer stack (blocks of 32) best over 1.6-1.8 (184 us), long-context (64) and ragged
// (16-64) over 2.1-2.4 and at 2.3 (173, 746 us).
constexpr double kMergePageCost32 = 1.7;
constexpr double kMergePageCost64 = 2.3;
constexpr int kMaxBatch = 512;

template <int D>
struct StreamCfg {
  static constexpr int TB = tile_bytes<D>();  // bf16 64 x D
  static constexpr int OB = 64 * D * 2;       // fp16 O~ / l page, laid out like a query tile
  // block role: K/V ring | 128-row query tile | two 128 x 64 score-probability tiles
  static constexpr int kKStages = 5;
  static constexpr int KStage = 2 * TB;
  static constexpr int off_qb = kKStages * KStage;
  static constexpr int QB = 2 * TB;  // 128 rows x D
  static constexpr int off_p = off_qb + QB;
  // two P tiles (128 rows x 64 keys bf16, 16 KB each), the second 8 KB after the first: only
  // rows 0-63 are ever written, and the rows of one tile that overlap the other only reach
  // rows of O that are never read
  static constexpr int PB = 128 * 128;
  static constexpr int kPOff = 8192;
  static constexpr int kBlockSmem = off_p + kPOff + PB;
  // merge role: query page | O~ / l page | m | l ring, then the gathered block keys / values
  static constexpr int kMStages = 5;
  static constexpr int MStage = TB + OB + 1024;
  static constexpr int off_kc = kMStages * MStage;
  static constexpr int off_vc = off_kc + TB;
  static constexpr int kMergeSmem = off_vc + TB;
  static constexpr int kSmem = (kBlockSmem > kMergeSmem ? kBlockSmem : kMergeSmem) + 1024;  // + alignment slack
  // tensor memory of the block role: O of softmax group 0 and of group 1 (D columns each),
  // then a score buffer of 64 columns per group
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 2 * D;
};

struct Shared {
  // A ring stage is shared by several consumer groups (pages go to the groups in turn),
  // so each (group, stage) has its own "full" barrier: a waiter must see every phase of
  // the barrier it waits on, since a parity wait cannot tell phase p from phase p + 2
  // (with one barrier per stage a group would skip the other groups' phases and could
  // take a stale stage whenever loads complete out of order).
  uint64_t full[3][5], empty[5], qfull, qempty;  // full: [group][stage] (block role: groups 0-1)
  uint64_t sfull[2], sempty[2], pfull[2], pvdone[2], ofinal, oempty;  // block role: MMA <-> softmax warps
  uint32_t tmem_base;
  float xmax[2][2][4][32];  // block role: [group][page parity][warp of the group][lane] maxima over the warp's keys
  float xm[2][64];          // block role: [group][query row] reference max at the end of a (b, h)
  float xl[8][32];          // block role: [warp][lane] sum over the warp's keys at the end of a (b, h)
  int abort_flag;
  int last_page[5];            // merge role: the last page issued into each stage (-1: none)
  int n_seq_units[kMaxBatch];  // H * pages of sequence b (0: invalid metadata)
  int cu[kMaxBatch + 1];       // unit prefix
};

__device__ __forceinline__ long long split_begin(long long c, long long U, long long G) { return c * U / G; }

// The first (b, h) pair, in (sequence, head) order, whose first unit (page) is at or after
// unit x: the units of (b, h) start at cu[b] + h * (units of b) / H.  Block-role CTA c owns
// the pairs that start in [c U / G, (c + 1) U / G), so every CTA of the role gets about the
// same number of pages (pairs of long sequences count for more than short ones).
__device__ __forceinline__ long long first_pair_at(const Shared& S, int batch, int H, long long x) {
  if (x >= S.cu[batch]) return static_cast<long long>(batch) * H;
  int lo = 0, hi = batch - 1;  // the sequence holding unit x: the smallest b with cu[b + 1] > x
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (S.cu[mid + 1] > x)
      hi = mid;
    else
      lo = mid + 1;
  }
  const long long np = S.n_seq_units[lo] / H;  // > 0: the sequence holds unit x
  const long long h = (x - S.cu[lo] + np - 1) / np;
  return static_cast<long long>(lo) * H + h;  // h == H is the next sequence's head 0
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


// ---------------------------------------------------------------------------
// Block role on the 5th-generation tensor cores.  For each (b, h) the CTA
// owns, the block queries stay in shared memory as a 128-row MMA tile and the
// pages go alternately to two softmax groups of four warps (group g takes the
// pages j with j mod 2 == g), each with its own online-softmax state
// (LaCache Eq. (2)-(6)): a reference max and running sums per row and its own
// O accumulator O_g in TMEM.  Per page of group g, warp 8 (g = 0) or 10
// (g = 1) issues S = Q K^T (M = 128, N = 64) into the group's TMEM score
// buffer; the group's warps write P = 2^(S - m_ref) as bf16 into the group's
// P tile, and warp 11 issues O_g += P V (M = 128, N = D, V as an MN-major
// operand), for both groups in page order.  The reference max is raised (O_g
// and the sums rescaled) only when a page's max exceeds it by more than 2^8,
// so every P stays <= 2^8 and the result is exact for any reference.  At the
// end of the (b, h) the two groups' states are merged exactly (the merge rule
// of LaCache §3.3.3) and O / l and L = m + log2 l are written.  Warp 9
// streams the tiles.
//
// A TMEM lane quadrant q is read only by warps q mod 4, which all issue from
// scheduler q, so the block queries (<= 32 or <= 64 rows) are loaded into
// every quadrant of the 128-row query tile (4 or 2 copies; the extra MMA rows
// cost nothing): warp q of a group reads its quadrant's copy and takes 1/4 or
// 1/2 of every page's keys, so the four schedulers share each page's softmax
// and each scheduler hosts one warp of either group.  A row's page max is
// exchanged within the group through shared memory once per page.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void block_role_tc(Shared& S, uint8_t* smem, const CUtensorMap& tm_qb,
                                              const CUtensorMap& tm_qb64, const CUtensorMap& tm_k,
                                              const CUtensorMap& tm_v, const AttnArgs& a,
                                              long long bh0, long long bh1) {
  using C = StreamCfg<D>;
  constexpr int TB = C::TB;
  constexpr float kRescale = 8.f;  // log2 units
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  uint8_t* ring = smem;
  uint8_t* q_tile = smem + C::off_qb;
  uint8_t* p_tile = smem + C::off_p;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {  // per softmax group
      mbar_init(&S.sfull[i], 1);   // the Q K^T commit
      mbar_init(&S.sempty[i], 4);  // the group's warps
      mbar_init(&S.pfull[i], 4);   // the group's warps
      mbar_init(&S.pvdone[i], 1);  // the P V commit
    }
    mbar_init(&S.ofinal, 1);
    mbar_init(&S.oempty, 8);  // the eight softmax warps
    fence_barrier_init();
  }
  if (warp == 8) tmem_alloc(&S.tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // a page is read once per step
      int nk = 0, nq = 0;
      int loads[2 * C::kKStages] = {};  // loads per (group, stage) "full" barrier
      bool waited = false;  // griddepcontrol.wait done
      for (long long bh = bh0; bh < bh1; ++bh) {
        const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
        const SeqMeta sm = load_meta(bt, b);
        if (!sm.ok) continue;
        const int np = (sm.nb + kPage - 1) / kPage;
        if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
        // the queries of (b, h) come from the preceding kernel; before them, the
        // first (b, h) streams its pages that hold no block rows into the free stages
        int p = 0;
        if (!waited) {
          for (; p < np && nk < C::kKStages; ++p, ++nk) {
            if (p * kPage < sm.sb + sm.bb && (p + 1) * kPage > sm.sb) break;  // a page with block rows
            const int y = (page_of(bt, b, p) * H + h) * kPage;
            uint8_t* kt = ring + nk * C::KStage;
            uint64_t* fb = &S.full[p & 1][nk];
            ++loads[(p & 1) * C::kKStages + nk];
            mbar_arrive_expect_tx(fb, 2 * TB);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf) {
              tma_load_2d_hint(kt + hf * 8192, &tm_k, fb, hf * 64, y, pol);
              tma_load_2d_hint(kt + TB + hf * 8192, &tm_v, fb, hf * 64, y, pol);
            }
          }
          griddep_wait();
          waited = true;
        }
        if (nq >= 1) wait_or_abort(S, &S.qempty, (nq - 1) & 1, bt.err);  // the previous (b, h)'s Q K^T are done
        mbar_arrive_expect_tx(&S.qfull, C::QB);
        {
          const bool wide = sm.bb > 32;  // copies of 64 rows (2) or 32 rows (4)
          const int rows = wide ? 64 : 32;
          for (int cp = 0; cp < 128 / rows; ++cp)
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              tma_load_3d(q_tile + hf * 16384 + cp * rows * 128, wide ? &tm_qb64 : &tm_qb, &S.qfull, hf * 64, h,
                          sm.cub);
        }
        ++nq;
        int raw_next = p < np ? page_raw(bt, b, p) : 0;  // loaded one page ahead of its use
        for (; p < np; ++p, ++nk) {
          const int raw = raw_next;
          if (p + 1 < np) raw_next = page_raw(bt, b, p + 1);
          const int s = nk % C::kKStages;
          if (nk >= C::kKStages) wait_or_abort(S, &S.empty[s], (nk / C::kKStages - 1) & 1, bt.err);
          const int y = (page_checked(bt, raw) * H + h) * kPage;
          uint8_t* kt = ring + s * C::KStage;
          uint64_t* fb = &S.full[p & 1][s];
          ++loads[(p & 1) * C::kKStages + s];
          mbar_arrive_expect_tx(fb, 2 * TB);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_2d_hint(kt + hf * 8192, &tm_k, fb, hf * 64, y, pol);
            tma_load_2d_hint(kt + TB + hf * 8192, &tm_v, fb, hf * 64, y, pol);
          }
        }
      }
      for (int i = 0; i < 2 * C::kKStages; ++i)  // every copy has landed: the last phase of each barrier
        if (loads[i] > 0 && !mbar_wait(&S.full[i / C::kKStages][i % C::kKStages], (loads[i] - 1) & 1))
          report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.qfull, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
      // Tail: the MMA issuers' last commits on the stages (Q K^T and P V) and on the
      // query tile have arrived, so no asynchronous arrival reaches this CTA's shared
      // memory after it exits (the next kernel's CTA may start on this SM at once).
      for (int i = (nk > C::kKStages ? nk - C::kKStages : 0); i < nk; ++i)
        if (!mbar_wait(&S.empty[i % C::kKStages], (i / C::kKStages) & 1)) report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.qempty, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ Q K^T issuers
    // An MMA issue takes tens of ns here, so the score MMAs of the two groups
    // and the P V MMAs have their own threads.  A K/V stage is free once its
    // Q K^T and its P V have completed (two commits); the query tile once both
    // score issuers have committed the (b, h)'s last MMAs.
    if (lane == 0) {
      constexpr uint32_t kIdS = umma_idesc_bf16(128, 64);
      const int g = warp == 8 ? 0 : 1;
      int n0 = 0, k = 0, nq = 0;  // pages of earlier (b, h) pairs, the group's pages so far, (b, h) pairs
      int uses[C::kKStages] = {};  // pages of this group taken from each stage so far
      for (long long bh = bh0; bh < bh1; ++bh) {
        const int b = static_cast<int>(bh / H);
        const SeqMeta sm = load_meta(bt, b);
        if (!sm.ok) continue;
        const int np = (sm.nb + kPage - 1) / kPage;
        wait_or_abort(S, &S.qfull, nq & 1, bt.err);
        tc_fence_after();
        const uint32_t qa = smem_u32(q_tile);
        for (int j = g; j < np; j += 2, ++k) {
          const int n = n0 + j, st = n % C::kKStages;
          wait_or_abort(S, &S.full[g][st], uses[st]++ & 1, bt.err);
          if (k >= 1) wait_or_abort(S, &S.sempty[g], (k - 1) & 1, bt.err);  // the group has read its last scores
          tc_fence_after();
          const uint32_t ka = smem_u32(ring + st * C::KStage);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16(tmem + C::kTmemS + g * 64, umma_desc_sw128(qa + (kk >> 2) * 16384 + (kk & 3) * 32),
                      umma_desc_sw128(ka + (kk >> 2) * 8192 + (kk & 3) * 32), kIdS, kk > 0 ? 1u : 0u);
          umma_commit(&S.sfull[g]);
          umma_commit(&S.empty[st]);  // K of the stage read
        }
        umma_commit(&S.qempty);  // this issuer no longer reads the (b, h)'s queries
        n0 += np;
        ++nq;
      }
    }
    __syncwarp();
  } else if (warp == 11) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      constexpr uint32_t kIdO = umma_idesc_bf16_bmn(128, D);
      int n = 0, nq = 0, k0 = 0, k1 = 0;  // pages, (b, h) pairs, each group's pages so far
      for (long long bh = bh0; bh < bh1; ++bh) {
        const int b = static_cast<int>(bh / H);
        const SeqMeta sm = load_meta(bt, b);
        if (!sm.ok) continue;
        const int np = (sm.nb + kPage - 1) / kPage;
        if (nq >= 1) wait_or_abort(S, &S.oempty, (nq - 1) & 1, bt.err);  // the previous (b, h)'s O read out
        for (int j = 0; j < np; ++j, ++n) {  // O_g += P V for page j (its stage landed before its scores)
          const int g = j & 1, st = n % C::kKStages;
          const int k = g == 0 ? k0++ : k1++;
          wait_or_abort(S, &S.pfull[g], k & 1, bt.err);
          tc_fence_after();
          const uint32_t pa = smem_u32(p_tile + g * C::kPOff);
          const uint32_t va = smem_u32(ring + st * C::KStage + TB);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + g * D, umma_desc_sw128(pa + kk * 32), umma_desc_sw128_mn(va + kk * 2048, 8192), kIdO,
                      (j > g || kk > 0) ? 1u : 0u);
          umma_commit(&S.empty[st]);  // V of the stage read
          umma_commit(&S.pvdone[g]);  // the group's P tile free, O_g holds page j
        }
        umma_commit(&S.ofinal);
        ++nq;
      }
      // Tail: this thread's last commits (each group's last P V, the last (b, h)) have
      // arrived before the CTA can exit.
      if (k0 >= 1 && !mbar_wait(&S.pvdone[0], (k0 - 1) & 1)) report_error(bt.err, kErrTimeout);
      if (k1 >= 1 && !mbar_wait(&S.pvdone[1], (k1 - 1) & 1)) report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.ofinal, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warps
    const int g = warp >> 2, wq = warp & 3;  // group, warp of the group (= TMEM lane quadrant)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
    uint8_t* p_own = p_tile + g * C::kPOff;
    int k = 0, nq = 0;  // the group's pages so far, (b, h) pairs
    for (long long bh = bh0; bh < bh1; ++bh) {
      const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
      const SeqMeta sm = load_meta(bt, b);
      if (!sm.ok) continue;
      const int np = (sm.nb + kPage - 1) / kPage;
      const int RQ = sm.bb > 32 ? 2 : 1;        // quadrants per copy of the queries
      const int rb = wq % RQ, slice = wq / RQ;  // row block, key slice
      const int KW = 16 * RQ;                   // keys per warp per page
      const int r = rb * 32 + lane;             // query row
      const bool row_ok = r < sm.bb;
      float m_ref = neg_inf(), l = 0.f;  // l: over this warp's keys
      for (int j = g; j < np; j += 2, ++k) {  // the group's pages (the same for its four warps)
        wait_or_abort(S, &S.sfull[g], k & 1, bt.err);
        tc_fence_after();
        float sc[32];
        const uint32_t scol = lane_base + C::kTmemS + g * 64 + slice * KW;
        if (RQ == 1)
          tmem_ld_32x32b_x16(scol, *reinterpret_cast<float(*)[16]>(sc));
        else
          tmem_ld_32x32b_x32(scol, sc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.sempty[g]);
        // scale, mask keys past the sequence, this warp's max; the row's page max
        const int nvalid = sm.nb - j * kPage - slice * KW;
        float mx4[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c >= KW) break;
          sc[c] = c < nvalid ? sc[c] * a.scale_log2 : neg_inf();
          mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
        }
        S.xmax[g][k & 1][wq][lane] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        if (g == 0)
          named_barrier(4, 128);
        else
          named_barrier(5, 128);
        float mx = neg_inf();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (q % RQ == rb) mx = fmaxf(mx, S.xmax[g][k & 1][q][lane]);
        // a new reference max (the group's first page, or a rise beyond the threshold) rescales
        // O_g and l; every warp of the row takes the same decision from the same values
        const bool first = j == g;
        const bool raise = row_ok && (first || mx > m_ref + kRescale);
        const float factor = raise && !first ? fast_exp2(m_ref - mx) : 1.f;
        if (raise) m_ref = mx;
        if (!first && __any_sync(0xffffffffu, factor != 1.f)) {
          l *= factor;
          if (slice == 0) {  // O_g's rows of this row block live in this warp's quadrant
            wait_or_abort(S, &S.pvdone[g], (k - 1) & 1, bt.err);  // O_g holds the group's earlier pages
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              float ov[32];
              tmem_ld_32x32b_x32(lane_base + g * D + c0, ov);
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] *= factor;
              tmem_st_32x32b_x32(lane_base + g * D + c0, ov);
            }
            tmem_st_wait();
          }
        }
        // P = 2^(S - m_ref) as bf16 into this warp's keys of row r of the group's P tile
        // (K-major, 128-byte swizzle), once the group's previous P V has read the tile
        if (k >= 1) wait_or_abort(S, &S.pvdone[g], (k - 1) & 1, bt.err);
        const float mu = row_ok ? m_ref : 0.f;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (cc * 8 >= KW) break;
          float pv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pv[e] = row_ok ? fast_exp2(sc[cc * 8 + e] - mu) : 0.f;
            l4[e & 3] += pv[e];
          }
          uint4 u;
          u.x = pack_bf16x2(pv[0], pv[1]);
          u.y = pack_bf16x2(pv[2], pv[3]);
          u.z = pack_bf16x2(pv[4], pv[5]);
          u.w = pack_bf16x2(pv[6], pv[7]);
          *reinterpret_cast<uint4*>(p_own + sw128_offset(r, slice * (KW / 8) + cc)) = u;
        }
        l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P visible to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pfull[g]);
      }
      // ---- the (b, h) is complete: merge the groups' states, O / l out, release O.  A row's
      // O_0 and O_1 live in the same TMEM lanes, so the warps of group 0 that hold the row
      // read both; only the maxima and sums go through shared memory.
      const bool has1 = np > 1;  // group 1 has pages
      if (slice == 0) S.xm[g][r] = m_ref;
      S.xl[warp][lane] = l;
      named_barrier(6, 256);
      if (g == 0 && slice == 0) {
        wait_or_abort(S, &S.ofinal, nq & 1, bt.err);
        tc_fence_after();
        float w0 = 0.f, w1 = 0.f, inv = 0.f, M = 0.f, L = 1.f;
        if (row_ok) {
          float lg[2] = {0.f, 0.f};  // each group's sum for row r
#pragma unroll
          for (int gg = 0; gg < 2; ++gg)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (q % RQ == rb) lg[gg] += S.xl[gg * 4 + q][lane];
          const float m0 = S.xm[0][r], m1 = has1 ? S.xm[1][r] : neg_inf();
          M = fmaxf(m0, m1);
          w0 = fast_exp2(m0 - M);
          w1 = has1 ? fast_exp2(m1 - M) : 0.f;
          L = w0 * lg[0] + w1 * lg[1];
          inv = 1.f / L;
          w0 *= inv;
          w1 *= inv;
        }
        const size_t orow = (static_cast<size_t>(sm.cus + sm.sb + r) * H + h);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float ov[32], ow[32];
          tmem_ld_32x32b_x32(lane_base + c0, ov);
          if (has1)
            tmem_ld_32x32b_x32(lane_base + D + c0, ow);
          else
#pragma unroll
            for (int i = 0; i < 32; ++i) ow[i] = 0.f;
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(of + orow * D + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float v[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) v[e] = ov[q * 8 + e] * w0 + ow[q * 8 + e] * w1;
              uint4 u;
              u.x = pack_bf16x2(v[0], v[1]);
              u.y = pack_bf16x2(v[2], v[3]);
              u.z = pack_bf16x2(v[4], v[5]);
              u.w = pack_bf16x2(v[6], v[7]);
              dst[q] = u;
            }
          }
        }
        if (row_ok && a.lse != nullptr) a.lse[orow] = (M + log2f(L)) * kLn2;
      }
      named_barrier(6, 256);  // xm and xl are read before the next (b, h) writes them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.oempty);
      ++nq;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_stream_kernel(
    const __grid_constant__ CUtensorMap tm_qb, const __grid_constant__ CUtensorMap tm_qb64,
    const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_o, const AttnArgs a, int n_block_ctas, int n_merge_ctas) {
  using C = StreamCfg<D>;
  constexpr int TB = C::TB;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ Shared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  const bool block_role = static_cast<int>(blockIdx.x) < n_block_ctas;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 5; ++s) {
      mbar_init(&S.full[0][s], 1);
      mbar_init(&S.full[1][s], 1);
      mbar_init(&S.full[2][s], 1);
      mbar_init(&S.empty[s], 2);  // block role: the Q K^T and P V completions
      S.last_page[s] = -1;
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 2);  // block role: the Q K^T completions of a (b, h) (two issuers)
    S.abort_flag = 0;
    fence_barrier_init();
  }
  // Programmatic dependent launch.  The preceding kernel (the step's projection)
  // writes q_block and the current blocks' k/v rows only, so the metadata, the
  // block table, the cached state and every other page are read before
  // griddepcontrol.wait (a precondition of the ABI); q_block and the pages that
  // hold block rows are read after it.
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
  // Block role: CTA c owns the (b, h) pairs, whole, that start in the units
  // [c U / G, (c + 1) U / G) (about U / G pages each).  Merge role: CTA c owns the
  // units [c U / G, (c + 1) U / G).
  const long long U = S.cu[bt.batch];
  const long long n_role = block_role ? n_block_ctas : n_merge_ctas;
  const long long c = block_role ? blockIdx.x : blockIdx.x - n_block_ctas;
  if (block_role) {
    const long long bh0 = first_pair_at(S, bt.batch, H, split_begin(c, U, n_role));
    const long long bh1 = first_pair_at(S, bt.batch, H, split_begin(c + 1, U, n_role));
    if (bh0 >= bh1) return;  // no pair starts in this CTA's range (uniform across the CTA)
    block_role_tc<D>(S, smem, tm_qb, tm_qb64, tm_k, tm_v, a, bh0, bh1);
    return;
  }
  const long long G = U < n_role ? U : n_role;
  if (c >= G) return;  // uniform across the CTA
  UWalk w;
  w.u = split_begin(c, U, G);
  w.u1 = split_begin(c + 1, U, G);
  w.seek(S, bt, H);

  // ===================================================================== merge role
  // Three groups of four warps take the pages with invariant rows in turn, page j (in walk
  // order) to group j % 3, through a ring of kMStages stages, page j in stage
  // j % kMStages; (group, stage) barrier phase j / (3 kMStages) is page j.  The stage of
  // page j is refilled with page j + kMStages by the leader of the group that consumed
  // page j, once its four warps are done with it.  Within a stage, issue, landing and
  // consumption therefore alternate: no barrier is armed again before its earlier phase
  // completed, and a group waits for its next phase of a barrier only after the previous.
  constexpr int NG = 3;
  uint8_t* ring = smem;
  uint8_t* kc_tile = smem + C::off_kc;
  uint8_t* vc_tile = smem + C::off_vc;
  const int grp = warp >> 2, mw = warp & 3;
  const bool leader = mw == 0 && lane == 0;
  const uint64_t pol = l2_evict_first_policy();  // the cached state is read once per step
  auto next_u = [&](UWalk& x) {                  // the next page with invariant rows
    do {
      x.next(S, bt, H);
    } while (x.valid() && !x.has_u_rows());
  };
  auto issue = [&](const UWalk& x, int raw, int j) {  // raw: the page's block-table entry
    const int s = j % C::kMStages;
    const int y = (page_checked(bt, raw) * H + x.h) * kPage;
    uint8_t* mt = ring + s * C::MStage;
    uint64_t* fb = &S.full[j % NG][s];
    S.last_page[s] = j;
    mbar_arrive_expect_tx(fb, TB + C::OB + 512);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) tma_load_2d_hint(mt + hf * 8192, &tm_q, fb, hf * 64, y, pol);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) tma_load_2d_hint(mt + TB + hf * 8192, &tm_o, fb, hf * 64, y, pol);
    bulk_load(mt + TB + C::OB, a.m_pool + y, 256, fb);
    bulk_load(mt + TB + C::OB + 256, a.l_pool + y, 256, fb);
  };
  // The leaders' look-ahead walkers: the page each group issues next (page grp + kMStages,
  // then every third page).  The first kMStages pages are issued here, before
  // griddepcontrol.wait (the cached state is not written by the preceding kernel).
  // Block-table entries are loaded ahead of their issue (all of the first kMStages at once,
  // then each leader's next one right after its current issue).
  UWalk wa = w;
  int wa_raw = 0;
  if (leader) {
    if (!wa.has_u_rows()) next_u(wa);
    if (grp == 0) {
      int raws[C::kMStages];
      UWalk x = wa;
#pragma unroll
      for (int j = 0; j < C::kMStages; ++j) {
        raws[j] = x.valid() ? page_raw(bt, x.b, x.p) : 0;
        if (x.valid()) next_u(x);
      }
#pragma unroll
      for (int j = 0; j < C::kMStages; ++j)
        if (wa.valid()) {
          issue(wa, raws[j], j);
          next_u(wa);
        }
    } else {
      for (int j = 0; j < C::kMStages + grp && wa.valid(); ++j) next_u(wa);
    }
    if (wa.valid()) wa_raw = page_raw(bt, wa.b, wa.p);
  }
  const float log2e = 1.4426950408889634f;
  int nm = 0;  // pages with invariant rows seen so far (every group counts all of them)
  int nkc = 32;
  __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
  for (; w.valid(); w.next(S, bt, H)) {
    if (w.seg_start()) {  // gather the fresh block keys / values of (b, h) through the table
      griddep_wait();               // they come from the preceding kernel (a no-op after the first time)
      named_barrier(2, kThreads);   // every group is done with the previous (b, h)'s
      nkc = w.sm.bb <= 32 ? 32 : 64;  // keys the QK^T below covers; rows past bb are zero
      const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
      const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
      for (int e = threadIdx.x; e < nkc * (D / 8); e += kThreads) {
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
      named_barrier(2, kThreads);
    }
    if (!w.has_u_rows()) continue;
    const int j = nm++;
    if (j % NG != grp) continue;  // another group's page
    const int s = j % C::kMStages;
    wait_or_abort(S, &S.full[grp][s], (j / (NG * C::kMStages)) & 1, bt.err);
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
      attend<D, 32, true>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
    else
      attend<D, 64, true>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
    st.reduce_l();
    // exact merge with the cached state (O~_c = l_c times the stored O~_c / l_c): the weights
    // of rows g and g + 8, then O~_c / l_c read in the accumulator layout (ldmatrix: rows g,
    // g + 8 of the 8-column tiles 2kk, 2kk + 1) and the merged rows staged the same way
    // (stmatrix) as bf16 in this warp's 16 rows of the q tile (read into registers above)
    const int r_lo = w.p * kPage, c_lo = w.sm.sb, c_hi = w.sm.sb + w.sm.bb;
    float wcl[2], wni[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = mw * 16 + (lane >> 2) + 8 * hr;
      const float mc = m_s[r] * log2e;  // cached max, base-2 units
      const float mn = st.m[hr];
      const float M = fmaxf(mc, mn);
      const float wc = mc == neg_inf() ? 0.f : fast_exp2(mc - M);
      const float wn = mn == neg_inf() ? 0.f : fast_exp2(mn - M);
      const float lc = l_s[r];
      const float L = wc * lc + wn * st.l[hr];
      const float inv = 1.f / L;
      wcl[hr] = wc * lc * inv;
      wni[hr] = wn * inv;
      const int pos = r_lo + r;
      if (a.lse != nullptr && (lane & 3) == 0 && pos < w.sm.nb && (pos < c_lo || pos >= c_hi))
        a.lse[static_cast<size_t>(w.sm.cus + pos) * H + w.h] = (M + __log2f(L)) * kLn2;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = tile_off(mw * 16 + (lane & 15), 2 * kk + (lane >> 4));
      uint32_t oc[4], out[4];
      ldmatrix_x4(oc, smem_u32(o_tile) + off);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const __half2 h2 = *reinterpret_cast<const __half2*>(&oc[2 * jj + hr]);
          const float* on = st.o[2 * kk + jj];
          out[2 * jj + hr] = pack_bf16x2(wcl[hr] * __low2float(h2) + wni[hr] * on[2 * hr],
                                         wcl[hr] * __high2float(h2) + wni[hr] * on[2 * hr + 1]);
        }
      stmatrix_x4(smem_u32(q_tile) + off, out);
    }
    __syncwarp();
    for (int e = lane; e < 16 * (D / 8); e += 32) {  // coalesced store of this warp's 16 rows
      const int r = mw * 16 + e / (D / 8), ch = e % (D / 8);
      const int pos = r_lo + r;
      if (pos >= w.sm.nb || (pos >= c_lo && pos < c_hi)) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(q_tile + tile_off(r, ch));
      *reinterpret_cast<uint4*>(of + (static_cast<size_t>(w.sm.cus + pos) * H + w.h) * D + ch * 8) = v;
    }
    // the stage's generic reads and writes before the TMA that refills it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    named_barrier(3 + grp, 128);  // the group's four warps are done with stage s
    if (leader && wa.valid() && !*reinterpret_cast<volatile int*>(&S.abort_flag)) {
      issue(wa, wa_raw, j + C::kMStages);
      for (int i = 0; i < NG && wa.valid(); ++i) next_u(wa);
      if (wa.valid()) wa_raw = page_raw(bt, wa.b, wa.p);
    }
  }
  // every issued copy has landed before the CTA exits (they all have, unless a wait gave up)
  named_barrier(2, kThreads);
  if (threadIdx.x == 0)
    for (int st = 0; st < C::kMStages; ++st) {
      const int j = S.last_page[st];
      if (j >= 0 && !mbar_wait(&S.full[j % NG][st], (j / (NG * C::kMStages)) & 1)) report_error(bt.err, kErrTimeout);
    }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  PoolMaps m;
  const bool merge = plan.n_merge_ctas > 0, block = plan.n_block_ctas > 0;
  cudaError_t e = encode_pool_maps(a, merge, merge, &m);
  if (e != cudaSuccess) return e;
  if (!merge) m.q = m.k, m.o = m.k;  // unused without the merge role
  CUtensorMap tm_qb = m.k, tm_qb64 = m.k;  // the block queries in boxes of 32 and of 64 rows
  if (block) {
    e = encode_3d_rows_sw128(&tm_qb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_block, D, a.n_heads,
                             a.bt.total_block_rows, 64, 32);
    if (e == cudaSuccess)
      e = encode_3d_rows_sw128(&tm_qb64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_block, D, a.n_heads,
                               a.bt.total_block_rows, 64, 64);
    if (e != cudaSuccess) return e;
  }
  constexpr int smem = StreamCfg<D>::kSmem;
  auto kern = attn_stream_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(plan.n_block_ctas + plan.n_merge_ctas), kThreads, smem, 0, stream, tm_qb, tm_qb64,
                    m.k, m.v, m.q, m.o, a, plan.n_block_ctas, plan.n_merge_ctas);
}


}  // namespace

AttnPlan attn_plan(int batch, int n_heads, int head_dim, int max_seq_len, int max_block_len, int total_seq_rows,
                   int total_block_rows, int num_sms, bool block, bool merge) {
  (void)head_dim;
  const double merge_cost = max_block_len <= 32 ? kMergePageCost32 : kMergePageCost64;
  AttnPlan p = {};
  const long long max_pages = (max_seq_len + kPage - 1) / kPage;
  const long long bh = static_cast<long long>(batch) * n_heads;
  const long long units = bh * max_pages;  // upper bound of the merge role's units
  const int g = static_cast<int>(units < num_sms ? (units < 1 ? 1 : units) : num_sms);
  if (block && merge) {
    // Split the CTAs between the roles by their work.  The block role walks every page of
    // every (sequence, head) and owns whole pairs, so with nb CTAs its time is about
    // ceil(pairs / nb) pairs of mean length; the merge role spreads the pages of the invariant
    // rows evenly, a merge page (query page, fp16 O~ / l page, row out) costing
    // merge_cost block pages.  Take the nb with the smallest larger of the two (in block
    // pages x 64), the most merge CTAs among equals.
    const double pair_rows = static_cast<double>(total_seq_rows) / batch;
    const double merge_rows = static_cast<double>(total_seq_rows - total_block_rows) * n_heads;
    const long long nb_max = std::min<long long>(bh, g - 1);
    long long best_nb = 1;
    double best = 0.0;
    for (long long nb = 1; nb <= nb_max; ++nb) {
      const double t = std::max(static_cast<double>((bh + nb - 1) / nb) * pair_rows,
                                merge_cost * merge_rows / static_cast<double>(g - nb));
      if (nb == 1 || t < best) {
        best = t;
        best_nb = nb;
      }
    }
    p.n_block_ctas = static_cast<int>(best_nb);
    p.n_merge_ctas = g - p.n_block_ctas < 1 ? 1 : g - p.n_block_ctas;
  } else {
    p.n_block_ctas = block ? static_cast<int>(bh < num_sms ? bh : num_sms) : 0;
    p.n_merge_ctas = merge ? g : 0;
  }
  return p;  // no workspace
}

bool attn_batch_supported(int batch) { return batch <= kMaxBatch; }

cudaError_t launch_step_attention(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (a.bt.batch <= 0 || plan.n_block_ctas + plan.n_merge_ctas == 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_d<128>(a, plan, stream) : launch_d<64>(a, plan, stream);
}

}  // namespace dllm
