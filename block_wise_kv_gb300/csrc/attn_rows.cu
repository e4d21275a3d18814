// attn_rows.cu — attention of 128-row query tiles on the 5th-generation tensor
// cores (sm_103a), in the modes of one persistent kernel.  Each mode gives,
// per sequence, the query rows (up to two position ranges) and the keys, in
// up to two phases:
//
//   kRowsState     the FACache build of a block boundary: every row r of U
//                  over the keys of U only, the online-softmax state
//                  (m, l, O~ / l) into m_pool / l_pool / o_pool (LaCache §3.3.3;
//                  Algorithm 1 with GenStep = True).
//   kRowsBlock     the block attention of blocks longer than one page: the
//                  block rows (from q_block) over every key of the sequence,
//                  O = O~ / l and L = m + ln l (Fast-dLLM DualCache "Inner step
//                  on block k", LaCache Eq. (2)-(6)).  This is the prefix-only
//                  cache mode of the Fast-dLLM page, where the block is the
//                  whole region after the prefix.
//   kRowsMerge     the FACache merge for such blocks: every row of U over the
//                  block keys, merged exactly with its cached state (LaCache
//                  §3.3.3, Algorithm 1 with GenStep = False).
//   kRowsStatePre  kRowsState, with the state of each row over the keys before
//                  the block (phase 1) also kept in the pre pools.
//   kRowsAdvOld,   the incremental block boundary (only the just-decoded
//   kRowsAdvNew    block's rows changed since the last one): the rows kept
//                  from the last boundary extend their pre state by the
//                  decoded block's keys (phase 1); the decoded rows build it
//                  over every key before the new block (phase 1); both then
//                  add the suffix keys (phase 2) for the state over U.
//
// In the modes with a pre state, the accumulator's state after phase 1 is
// written to the pre pools and accumulation goes on through phase 2; the kept
// rows of kRowsAdvOld start from their pre state, loaded into the accumulator
// (O_t, reference max, sum) before the first page, so that the exact merge
// (LaCache §3.3.3) of the pre state with the new keys' partial state is the
// online softmax itself.
//
// A unit of work is (sequence b, head h, a pair of query tiles): two tiles of
// 128 query rows that share every K/V page the unit streams.  Warp 9 streams
// the query tiles and the K/V pages (TMA, 128-byte swizzle) into an mbarrier
// ring; warps 8 (tile 0) and 10 (tile 1) issue, per page, S_t = Q_t K^T into
// one of two score buffers of tile t and then O_t += P_t V of the previous
// page (P_t from shared memory, V as an MN-major operand), with S, O in
// tensor memory; warps 0-3 (tile 0) and 4-7 (tile 1) run the softmax, one
// thread per query row (TMEM lane = row).  The reference max of a row is
// raised (its O row and sum rescaled) only when a page's max exceeds it by
// more than 2^8, so every P stays <= 2^8; the exact max is tracked beside it
// for the states' m.  Units are split over the CTAs by their K/V pages (every
// unit of a sequence streams the same pages), and a CTA walks its units in
// order, loading the next unit's query tiles while the current one finishes.
#include <math.h>

#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

constexpr int kThreads = 352;  // warps 0-7 softmax, 8 and 10 MMA issuers, 9 producer
constexpr int kMaxSeqs = 1024;  // sequences per launch (the host launches larger batches in slices)
constexpr float kRescale = 8.f;  // log2 units

template <int D>
struct RowsCfg {
  static constexpr int TB = tile_bytes<D>();  // bf16 64 rows x D
  static constexpr int QB = 2 * TB;           // one 128-row query tile
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int KVB = 2 * TB;          // a K page and a V page
  static constexpr int off_q = 0;             // two query tiles
  static constexpr int off_kv = 2 * QB;
  static constexpr int off_p = off_kv + kStages * KVB;  // two P tiles (128 x 64 bf16)
  static constexpr int PB = 128 * 128;
  static constexpr int kSmem = off_p + 2 * PB + 1024;  // + alignment slack
  // tensor memory: O_0, O_1 (D columns each), then four 64-column score buffers
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 256;
};

struct RowsShared {
  uint64_t kvfull[6], kvempty[6], qfull, qempty;
  uint64_t sfull[2][2], sfree[2][2], pfull[2], pfree[2], ofull[2], ofree[2];
  uint32_t tmem_base;
  int abort_flag;
  long long cu_units[kMaxSeqs + 1];  // unit prefix over the launch's sequences
  long long cu_cost[kMaxSeqs + 1];   // K/V page prefix (the cost of the units)
};

// Per-sequence shape of the work of one mode: the query rows, the query tiles
// (of 128 rows) that hold them, and the K/V pages (of 64 keys) of the two key
// phases.
struct RowsSeq {
  SeqMeta sm;
  int np;                  // pages of the sequence
  int r0, r1, r2, r3;      // query rows [r0, r1) u [r2, r3) (kRowsBlock: block rows, relative)
  int k0, k1, k2, k3;      // keys: phase 1 [k0, k1), phase 2 [k2, k3)
  int nq, ta0, na, tb0;    // query tiles: tile k -> k < na ? ta0 + k : tb0 + (k - na)
  int p1, n1, p2, n2, nk;  // key pages: p1 .. p1 + n1 - 1, then p2 .. p2 + n2 - 1
};

__device__ __forceinline__ SeqMeta load_meta_rows(const BatchArgs& bt, int b) {
  SeqMeta m;
  m.nb = __ldg(bt.seq_len + b);
  m.bb = __ldg(bt.block_len + b);
  m.sb = __ldg(bt.block_start + b);
  m.cub = __ldg(bt.cu_block + b);
  m.cus = __ldg(bt.cu_seq + b);
  m.ok = m.nb >= 1 && m.nb <= bt.max_seq_len && m.bb >= 1 && m.bb <= bt.max_block_len && m.sb >= 0 &&
         m.sb + m.bb <= m.nb && (m.nb + kPage - 1) / kPage <= bt.max_pages && m.cub >= 0 &&
         m.cub + m.bb <= bt.total_block_rows && m.cus >= 0 && m.cus + m.nb <= bt.total_seq_rows;
  return m;
}

__device__ __forceinline__ RowsSeq rows_seq(const AttnArgs& a, int b, int mode) {
  RowsSeq s;
  s.sm = load_meta_rows(a.bt, b);
  s.np = s.nq = s.na = s.ta0 = s.tb0 = s.nk = s.n1 = s.n2 = s.p1 = s.p2 = 0;
  s.r0 = s.r1 = s.r2 = s.r3 = s.k0 = s.k1 = s.k2 = s.k3 = 0;
  if (!s.sm.ok) return s;
  const int nb = s.sm.nb, sb = s.sm.sb, ce = s.sm.sb + s.sm.bb;  // C = [sb, ce)
  int ps = 0;  // the decoded block [ps, sb)
  if (mode == kRowsAdvOld || mode == kRowsAdvNew) {
    ps = __ldg(a.prev_start + b);
    if (ps < 0 || ps >= sb) {
      s.sm.ok = false;
      return s;
    }
  }
  s.np = (nb + kPage - 1) / kPage;
  switch (mode) {
    case kRowsBlock:  // the block rows over every key
      s.r0 = 0, s.r1 = s.sm.bb, s.k0 = 0, s.k1 = nb;
      break;
    case kRowsMerge:  // U over the keys of C
      s.r0 = 0, s.r1 = sb, s.r2 = ce, s.r3 = nb, s.k0 = sb, s.k1 = ce;
      break;
    case kRowsAdvOld:  // the rows kept: the decoded block's keys, then the suffix
      s.r0 = 0, s.r1 = ps, s.r2 = ce, s.r3 = nb, s.k0 = ps, s.k1 = sb, s.k2 = ce, s.k3 = nb;
      break;
    case kRowsAdvNew:  // the decoded rows: every key before the block, then the suffix
      s.r0 = ps, s.r1 = sb, s.k0 = 0, s.k1 = sb, s.k2 = ce, s.k3 = nb;
      break;
    default:  // kRowsState, kRowsStatePre: U over the prefix, then the suffix
      s.r0 = 0, s.r1 = sb, s.r2 = ce, s.r3 = nb, s.k0 = 0, s.k1 = sb, s.k2 = ce, s.k3 = nb;
      break;
  }
  // query tiles over the row ranges (kRowsBlock: tiles of the block rows)
  int ta1 = s.r1 > s.r0 ? (s.r1 + 127) / 128 : s.r0 / 128;
  int tb1 = s.r3 > s.r2 ? (s.r3 + 127) / 128 : s.r2 / 128;
  s.ta0 = s.r0 / 128;
  s.tb0 = s.r2 / 128;
  if (ta1 == s.ta0) {  // first range empty
    s.ta0 = s.tb0;
    ta1 = tb1;
    s.tb0 = tb1;
  } else {
    s.tb0 = max(s.tb0, ta1);
    tb1 = max(tb1, s.tb0);
  }
  s.na = ta1 - s.ta0;
  s.nq = s.na + (tb1 - s.tb0);
  // key pages of the two phases (a page may hold keys of both: it is streamed twice)
  if (s.k1 > s.k0) {
    s.p1 = s.k0 / kPage;
    s.n1 = (s.k1 + kPage - 1) / kPage - s.p1;
  }
  if (s.k3 > s.k2) {
    s.p2 = s.k2 / kPage;
    s.n2 = (s.k3 + kPage - 1) / kPage - s.p2;
  }
  s.nk = s.n1 + s.n2;
  return s;
}

// The i-th K/V page of a unit of sequence s, and the key range of its phase.
__device__ __forceinline__ int key_page(const RowsSeq& s, int i) { return i < s.n1 ? s.p1 + i : s.p2 + (i - s.n1); }

// The first unit, in unit order, whose first page is at or after page x of the launch's
// cost (K/V pages): CTA c owns the units that start in [c W / G, (c + 1) W / G).  Every
// unit of a sequence streams the same pages.
__device__ __forceinline__ long long first_unit_at(const RowsShared& S, int nseq, long long x) {
  if (x >= S.cu_cost[nseq]) return S.cu_units[nseq];
  int lo = 0, hi = nseq - 1;  // the sequence holding page x: the smallest b with cu_cost[b + 1] > x
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (S.cu_cost[mid + 1] > x)
      hi = mid;
    else
      lo = mid + 1;
  }
  const long long nk = (S.cu_cost[lo + 1] - S.cu_cost[lo]) / (S.cu_units[lo + 1] - S.cu_units[lo]);
  return S.cu_units[lo] + (x - S.cu_cost[lo] + nk - 1) / nk;
}

// Walk over the units [u, u1): sequence, head, pair of query tiles.
struct RWalk {
  long long u, u1;
  int b, h, pr, npairs;
  RowsSeq s;
  __device__ __forceinline__ void seek(const RowsShared& S, const AttnArgs& a, int mode, int b_begin, int nseq,
                                       int H) {
    int lo = 0, hi = nseq - 1;  // the largest b with cu_units[b] <= u: skips sequences without units
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (S.cu_units[mid] <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    b = lo;
    s = rows_seq(a, b_begin + b, mode);
    npairs = static_cast<int>((S.cu_units[b + 1] - S.cu_units[b]) / H);
    const int r = static_cast<int>(u - S.cu_units[b]);
    h = r / npairs;
    pr = r % npairs;
  }
  __device__ __forceinline__ bool valid() const { return u < u1; }
  __device__ __forceinline__ void next(const RowsShared& S, const AttnArgs& a, int mode, int b_begin, int nseq,
                                       int H) {
    if (++u >= u1) return;
    if (++pr == npairs) {
      pr = 0;
      if (++h == H) seek(S, a, mode, b_begin, nseq, H);
    }
  }
  __device__ __forceinline__ bool has1() const { return 2 * pr + 1 < s.nq; }
  // tile index (of 128 rows) of query tile t of the unit
  __device__ __forceinline__ int tile(int t) const {
    const int k = 2 * pr + t;
    return k < s.na ? s.ta0 + k : s.tb0 + (k - s.na);
  }
};

// Bounded wait that gives up (and makes the whole CTA give up) after a timeout.
__device__ __forceinline__ void wait_or_abort(RowsShared& S, uint64_t* bar, uint32_t parity, int32_t* err) {
  if (*reinterpret_cast<volatile int*>(&S.abort_flag)) return;
  if (!mbar_wait(bar, parity)) {
    S.abort_flag = 1;
    report_error(err, kErrTimeout);
  }
}

// Write row srow of the accumulator's state to the pools (mo, lo, oo): m in
// natural units is the exact max m_true, l is taken from the reference max
// m_ref to m_true, and the state's O~ is kept normalised: oo = O~ / l (O_t's
// row at o_row over the row's sum; zero when !have_o or l = 0), as fp16.  O~ / l
// is a convex combination of value rows, so it stays within fp16's range unless
// a value does; a row beyond it flags kErrRange.  The O_t row is read by the
// whole warp (tcgen05.ld), the pools only for row_out.
template <int D>
__device__ __forceinline__ void store_state(uint32_t o_row, bool have_o, float m_ref, float m_true, float l,
                                            float* mo_p, float* lo_p, void* oo_p, size_t srow, bool row_out,
                                            int* err) {
  const float c = (!have_o || m_ref == neg_inf()) ? 0.f : fast_exp2(m_ref - m_true);
  const float inv = (have_o && l > 0.f) ? 1.f / l : 0.f;  // O~ / l: the rescale to m_true cancels
  if (row_out) {
    mo_p[srow] = m_true * kLn2;  // -inf stays -inf
    lo_p[srow] = l * c;
  }
  float amax = 0.f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 32) {
    float ov[32];
    if (have_o) {
      tmem_ld_32x32b_x32(o_row + c0, ov);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = 0.f;
    }
    if (row_out) {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        ov[e] *= inv;
        amax = fmaxf(amax, fabsf(ov[e]));
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(oo_p) + srow * D + c0);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        dst[qq] = make_uint4(pack_f16x2(ov[8 * qq], ov[8 * qq + 1]), pack_f16x2(ov[8 * qq + 2], ov[8 * qq + 3]),
                             pack_f16x2(ov[8 * qq + 4], ov[8 * qq + 5]), pack_f16x2(ov[8 * qq + 6], ov[8 * qq + 7]));
    }
  }
  if (row_out && !(amax <= 65504.f)) report_error(err, kErrRange);
}

// Eight fp16 (one 16-byte load) to fp32 times k.
__device__ __forceinline__ void f16x8_scaled(const uint4& u, float k, float* out) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    out[2 * i] = __low2float(h) * k;
    out[2 * i + 1] = __high2float(h) * k;
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    rows_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qb,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const AttnArgs a, int b_begin, int nseq) {
  using C = RowsCfg<D>;
  constexpr int TB = C::TB;
  constexpr int NST = C::kStages;
  // modes that keep the state after phase 1 in the pre pools
  constexpr bool kPre = MODE == kRowsStatePre || MODE == kRowsAdvOld || MODE == kRowsAdvNew;
  // the kept rows of an incremental boundary start from their pre state (loaded into O_t)
  constexpr bool kInit = MODE == kRowsAdvOld;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* q_tiles = smem + C::off_q;
  uint8_t* kv_ring = smem + C::off_kv;
  uint8_t* p_tiles = smem + C::off_p;
  __shared__ RowsShared S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&S.kvfull[s], 1);
      mbar_init(&S.kvempty[s], 2);  // a commit of each issuer after its last MMA that reads the stage
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 2);  // both issuers
    for (int t = 0; t < 2; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&S.sfull[t][b], 1);
        mbar_init(&S.sfree[t][b], 4);  // the tile's four softmax warps
      }
      mbar_init(&S.pfull[t], 4);
      mbar_init(&S.pfree[t], 1);
      mbar_init(&S.ofull[t], 1);
      mbar_init(&S.ofree[t], 4);
    }
    S.abort_flag = 0;
    fence_barrier_init();
  }
  // Units and their cost (K/V pages) per sequence, then their prefix sums (warp 0).
  for (int i = threadIdx.x; i < nseq; i += kThreads) {
    const RowsSeq s = rows_seq(a, b_begin + i, MODE);
    if (!s.sm.ok) report_error(bt.err, kErrBadShape);
    const long long units = s.nk > 0 && s.nq > 0 ? static_cast<long long>(H) * ((s.nq + 1) / 2) : 0;
    S.cu_units[i + 1] = units;
    S.cu_cost[i + 1] = units * s.nk;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (nseq + 31) / 32, i0 = lane * per, i1 = min(nseq, i0 + per);
    long long su = 0, sc = 0;
    for (int i = i0; i < i1; ++i) {
      su += S.cu_units[i + 1];
      sc += S.cu_cost[i + 1];
    }
    long long xu = su, xc = sc;  // inclusive scan over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long yu = __shfl_up_sync(0xffffffffu, xu, o), yc = __shfl_up_sync(0xffffffffu, xc, o);
      if (lane >= o) {
        xu += yu;
        xc += yc;
      }
    }
    long long ru = xu - su, rc = xc - sc;  // exclusive
    for (int i = i0; i < i1; ++i) {
      ru += S.cu_units[i + 1];
      rc += S.cu_cost[i + 1];
      S.cu_units[i + 1] = ru;
      S.cu_cost[i + 1] = rc;
    }
    if (lane == 0) {
      S.cu_units[0] = 0;
      S.cu_cost[0] = 0;
    }
  }
  if (warp == 8) tmem_alloc(&S.tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  griddep_launch_dependents();
  // Every read of the pools, q_block and the cached state comes after the preceding
  // kernel (the projection that writes them) has completed.
  griddep_wait();

  const long long W = S.cu_cost[nseq];
  const long long G = gridDim.x, c = blockIdx.x;
  RWalk w0;
  w0.u = first_unit_at(S, nseq, c * W / G);
  w0.u1 = first_unit_at(S, nseq, (c + 1) * W / G);
  if (w0.u < w0.u1) w0.seek(S, a, MODE, b_begin, nseq, H);

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int nkv = 0, nq = 0;
      for (RWalk w = w0; w.valid(); w.next(S, a, MODE, b_begin, nseq, H)) {
        if (*reinterpret_cast<volatile int*>(&S.abort_flag)) break;
        const int gb = b_begin + w.b;
        const int T = w.has1() ? 2 : 1;
        // the unit's query tiles, once the previous unit's score MMAs have read theirs
        if (nq >= 1) wait_or_abort(S, &S.qempty, (nq - 1) & 1, bt.err);
        mbar_arrive_expect_tx(&S.qfull, T * C::QB);
        for (int t = 0; t < T; ++t) {
          const int tq = w.tile(t);
          uint8_t* qt = q_tiles + t * C::QB;
          for (int cp = 0; cp < 2; ++cp) {  // two boxes of 64 rows
            if (MODE == kRowsBlock) {
              // block rows cu_block[b] + 128 tq + 64 cp ...: rows past the end of q_block read as
              // zeros, rows of the next sequence are loaded but never written out
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf)
                tma_load_3d(qt + hf * 16384 + cp * 8192, &tm_qb, &S.qfull, hf * 64, w.h, w.s.sm.cub + 128 * tq + 64 * cp);
            } else {
              // page 2 tq + cp of the sequence (a tile's second page past the end repeats its
              // first: those rows are never written out)
              const int p = 2 * tq + cp < w.s.np ? 2 * tq + cp : 2 * tq;
              const int y = (page_of(bt, gb, p) * H + w.h) * kPage;
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(qt + hf * 16384 + cp * 8192, &tm_q, &S.qfull, hf * 64, y);
            }
          }
        }
        ++nq;
        for (int i = 0; i < w.s.nk; ++i, ++nkv) {
          const int st = nkv % NST;
          if (nkv >= NST) wait_or_abort(S, &S.kvempty[st], (nkv / NST - 1) & 1, bt.err);
          const int y = (page_of(bt, gb, key_page(w.s, i)) * H + w.h) * kPage;
          uint8_t* kt = kv_ring + st * C::KVB;
          mbar_arrive_expect_tx(&S.kvfull[st], C::KVB);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            tma_load_2d(kt + hf * 8192, &tm_k, &S.kvfull[st], hf * 64, y);
            tma_load_2d(kt + TB + hf * 8192, &tm_v, &S.kvfull[st], hf * 64, y);
          }
        }
      }
      // Tail: every copy has landed, and the MMA issuer's last commits on the stages and on
      // the query tiles have arrived, before the CTA can exit.
      for (int i = (nkv > NST ? nkv - NST : 0); i < nkv; ++i)
        if (!mbar_wait(&S.kvfull[i % NST], (i / NST) & 1)) report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.qfull, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
      for (int i = (nkv > NST ? nkv - NST : 0); i < nkv; ++i)
        if (!mbar_wait(&S.kvempty[i % NST], (i / NST) & 1)) report_error(bt.err, kErrTimeout);
      if (nq >= 1 && !mbar_wait(&S.qempty, (nq - 1) & 1)) report_error(bt.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per query tile t (warp 8: tile 0, warp 10: tile 1), so that neither
    // tile's MMAs wait for the other tile's softmax.  Per page i of a unit: S_t(i) =
    // Q_t K_i^T, then O_t += P_t(i-1) V_{i-1} (the scores of page i run while the softmax
    // of page i-1 finishes).  A stage is free once both issuers have committed its last
    // MMAs; the issuer of tile 1 walks (and releases) the pages of a unit without a
    // second tile too.
    if (lane == 0) {
      constexpr uint32_t kIdS = umma_idesc_bf16(128, 64);
      constexpr uint32_t kIdO = umma_idesc_bf16_bmn(128, D);
      const int t = warp == 8 ? 0 : 1;
      int nkv = 0, nq = 0, ns = 0, npv = 0, no = 0;  // stages, units, S buffers, P V, units of tile t
      const uint32_t qa = smem_u32(q_tiles + t * C::QB), ring0 = smem_u32(kv_ring);
      const uint32_t pa = smem_u32(p_tiles + t * C::PB);
      for (RWalk w = w0; w.valid(); w.next(S, a, MODE, b_begin, nseq, H)) {
        const bool mine = t == 0 || w.has1();
        const int nk = w.s.nk;
        wait_or_abort(S, &S.qfull, nq & 1, bt.err);
        tc_fence_after();
        // O_t += P_t V of page i (stage st); the unit's first overwrites O_t (adds to the pre
        // state loaded there, for the kept rows of an incremental boundary) once the softmax
        // warps have read the previous unit's O_t out
        auto pv = [&](int i, int st) {
          if (mine) {
            wait_or_abort(S, &S.pfull[t], npv & 1, bt.err);
            if (i == 0 && no >= 1) wait_or_abort(S, &S.ofree[t], (no - 1) & 1, bt.err);
            tc_fence_after();
            const uint32_t va = ring0 + st * C::KVB + TB;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + t * D, umma_desc_sw128(pa + kk * 32), umma_desc_sw128_mn(va + kk * 2048, 8192), kIdO,
                        (i > 0 || kInit || kk > 0) ? 1u : 0u);
            umma_commit(&S.pfree[t]);
            ++npv;
            if (i == nk - 1) {
              umma_commit(&S.ofull[t]);
              ++no;
            }
          }
          umma_commit(&S.kvempty[st]);  // this issuer's MMAs that read the stage have completed
        };
        int prev_st = 0;
        for (int i = 0; i < nk; ++i, ++nkv) {
          const int st = nkv % NST;
          wait_or_abort(S, &S.kvfull[st], (nkv / NST) & 1, bt.err);
          tc_fence_after();
          if (mine) {
            const int bsel = ns & 1;
            if (ns >= 2) wait_or_abort(S, &S.sfree[t][bsel], ((ns >> 1) - 1) & 1, bt.err);
            tc_fence_after();
            const uint32_t ka = ring0 + st * C::KVB;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_bf16(tmem + C::kTmemS + (2 * t + bsel) * 64,
                        umma_desc_sw128(qa + (kk >> 2) * 16384 + (kk & 3) * 32),
                        umma_desc_sw128(ka + (kk >> 2) * 8192 + (kk & 3) * 32), kIdS, kk > 0 ? 1u : 0u);
            umma_commit(&S.sfull[t][bsel]);
            ++ns;
          }
          if (i == nk - 1) umma_commit(&S.qempty);  // the unit's queries are no longer read
          if (i >= 1) pv(i - 1, prev_st);
          prev_st = st;
        }
        if (nk >= 1) pv(nk - 1, prev_st);
        ++nq;
      }
      // Tail: the last P V commit has arrived before the CTA can exit.
      if (npv >= 1 && !mbar_wait(&S.pfree[t], (npv - 1) & 1)) report_error(bt.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2, wq = warp & 3;  // query tile, warp of the tile (= TMEM lane quadrant)
    const int r = wq * 32 + lane;            // query row of the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t o_row = lane_base + t * D;  // this thread's row of O_t
    uint8_t* p_own = p_tiles + t * C::PB;
    int ns = 0, pw = 0, no = 0;  // S buffers read, P tiles written, units finished
    for (RWalk w = w0; w.valid(); w.next(S, a, MODE, b_begin, nseq, H)) {
      if (t == 1 && !w.has1()) continue;
      const RowsSeq& q = w.s;
      const int gb = b_begin + w.b;
      const int tq = w.tile(t);
      // the position of this thread's query row, whether it is written out, and its slot
      // in the pools
      int pos;
      bool row_out;
      if (MODE == kRowsBlock) {
        const int i = 128 * tq + r;
        pos = q.sm.sb + i;
        row_out = i < q.sm.bb;
      } else {
        pos = 128 * tq + r;
        row_out = (pos >= q.r0 && pos < q.r1) || (pos >= q.r2 && pos < q.r3);
      }
      size_t srow = 0;
      if (MODE != kRowsBlock && row_out)
        srow = (static_cast<size_t>(page_of(bt, gb, pos / kPage)) * H + w.h) * kPage + pos % kPage;
      float m_ref = neg_inf(), m_true = neg_inf(), l = 0.f;
      if (kInit) {
        // the kept row's pre state becomes the accumulator: O_t's row (the previous unit's
        // O_t is read out and its last P V complete), the reference max and the sum
        float mi = neg_inf(), li = 0.f;
        if (row_out) {
          mi = a.m_pre[srow] * 1.4426950408889634f;  // base-2 units
          li = a.l_pre[srow];
        }
        const bool have = mi != neg_inf();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {  // O~ = l * (O~ / l), 32 columns at a time
          float ov[32];
          if (have) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __half*>(a.o_pre) + srow * D + c0);
            const uint4 u0 = src[0], u1 = src[1], u2 = src[2], u3 = src[3];
            f16x8_scaled(u0, li, ov);
            f16x8_scaled(u1, li, ov + 8);
            f16x8_scaled(u2, li, ov + 16);
            f16x8_scaled(u3, li, ov + 24);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = 0.f;
          }
          tmem_st_32x32b_x32(o_row + c0, ov);
        }
        tmem_st_wait();
        if (have) {
          m_ref = mi;
          m_true = mi;
          l = li;
        }
      }
      if (kPre && q.n1 == 0)  // no phase 1: an empty pre state
        store_state<D>(o_row, false, m_ref, m_true, l, a.m_pre, a.l_pre, a.o_pre, srow, row_out, bt.err);
      for (int i = 0; i < q.nk; ++i) {
        const int bsel = ns & 1;
        wait_or_abort(S, &S.sfull[t][bsel], (ns >> 1) & 1, bt.err);
        tc_fence_after();
        float sc[64];
        tmem_ld_32x32b_x64(lane_base + C::kTmemS + (2 * t + bsel) * 64, sc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.sfree[t][bsel]);
        ++ns;
        // this row's page max over the keys of the page's phase (raw scores: the scale is
        // positive, so it is applied to the max and folded into the exponent below); a page
        // whose keys all belong to the phase takes the unmasked path (uniform per page)
        const bool ph2 = i >= q.n1;
        const int key0 = key_page(q, i) * kPage;
        const int klo = ph2 ? q.k2 : q.k0, khi = ph2 ? q.k3 : q.k1;
        if (!(key0 >= klo && key0 + kPage <= khi)) {
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (key0 + cc < klo || key0 + cc >= khi) sc[cc] = neg_inf();
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = sc[e];
#pragma unroll
        for (int cc = 8; cc < 64; ++cc) mx8[cc & 7] = fmaxf(mx8[cc & 7], sc[cc]);
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * a.scale_log2;
        // pre modes: the state after phase 1 (before this page) goes to the pre pools
        const bool snap = kPre && i == q.n1 && i > 0;
        const float s_mref = m_ref, s_mtrue = m_true, s_l = l;
        m_true = fmaxf(m_true, mx);
        // a new reference max (the accumulator's first keys, or a rise beyond the threshold)
        float factor = 1.f;
        if (m_ref == neg_inf()) {
          m_ref = mx;
        } else if (mx > m_ref + kRescale) {
          factor = fast_exp2(m_ref - mx);
          m_ref = mx;
        }
        const float mu = m_ref == neg_inf() ? 0.f : m_ref;
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) {
          sc[cc] = fast_exp2(fmaf(sc[cc], a.scale_log2, -mu));  // masked: 2^-inf = 0
          l8[cc & 7] += sc[cc];
        }
        l = l * factor + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
        // the tile's previous P V has completed: its P tile is free and O_t holds every
        // earlier page (rescaled here when the reference max rose)
        if (pw >= 1) wait_or_abort(S, &S.pfree[t], (pw - 1) & 1, bt.err);
        tc_fence_after();
        if (snap)  // O_t holds phase 1 (relative to the reference max before this page)
          store_state<D>(o_row, true, s_mref, s_mtrue, s_l, a.m_pre, a.l_pre, a.o_pre, srow, row_out, bt.err);
        if (__any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            tmem_ld_32x32b_x32(o_row + c0, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= factor;
            tmem_st_32x32b_x32(o_row + c0, ov);
          }
          tmem_st_wait();
        }
        // P = 2^(S - m_ref) as bf16 into row r of the tile's P tile (K-major, 128-byte swizzle)
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint4 u;
          u.x = pack_bf16x2(sc[8 * cc], sc[8 * cc + 1]);
          u.y = pack_bf16x2(sc[8 * cc + 2], sc[8 * cc + 3]);
          u.z = pack_bf16x2(sc[8 * cc + 4], sc[8 * cc + 5]);
          u.w = pack_bf16x2(sc[8 * cc + 6], sc[8 * cc + 7]);
          *reinterpret_cast<uint4*>(p_own + sw128_offset(r, cc)) = u;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P visible to the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.pfull[t]);
        ++pw;
      }
      // ---- the unit is complete for this tile: O_t out, then released for the next unit
      wait_or_abort(S, &S.ofull[t], no & 1, bt.err);
      tc_fence_after();
      if (MODE == kRowsState || kPre) {
        store_state<D>(o_row, true, m_ref, m_true, l, a.m_pool, a.l_pool, a.o_pool, srow, row_out, bt.err);
        if (kPre && q.n2 == 0)  // phase 1 only: the pre state is the same
          store_state<D>(o_row, true, m_ref, m_true, l, a.m_pre, a.l_pre, a.o_pre, srow, row_out, bt.err);
      } else {
        // O = (w_c O~_c + w_f O_t) / L with the cached state (merge) or O_t / l (block rows)
        float wc = 0.f, wf = 1.f, M = m_ref, L = l, lc = 0.f;
        if (MODE == kRowsMerge && row_out) {
          const float mc = __ldg(a.m_pool + srow) * 1.4426950408889634f;  // base-2 units
          lc = __ldg(a.l_pool + srow);
          M = fmaxf(mc, m_ref);
          wc = mc == neg_inf() ? 0.f : fast_exp2(mc - M);
          wf = fast_exp2(m_ref - M);
          L = wc * lc + wf * l;
        }
        const float inv = row_out ? 1.f / L : 0.f;
        wc *= inv;
        wf *= inv;
        const float wcl = wc * lc;  // the cached part's weight on O~_c / l_c
        const size_t orow = static_cast<size_t>(q.sm.cus + pos) * H + w.h;
        __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float ov[32];
          tmem_ld_32x32b_x32(o_row + c0, ov);
          if (row_out) {
            if (MODE == kRowsMerge) {  // wc l_c (O~_c / l_c) + wf O_t
              const uint4* oc = reinterpret_cast<const uint4*>(static_cast<const __half*>(a.o_pool) +
                                                               srow * D + c0);
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                float cv[8];
                f16x8_scaled(__ldg(oc + qq), wcl, cv);
#pragma unroll
                for (int e = 0; e < 8; ++e) ov[8 * qq + e] = cv[e] + wf * ov[8 * qq + e];
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) ov[e] *= wf;
            }
            uint4* dst = reinterpret_cast<uint4*>(of + orow * D + c0);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint4 u;
              u.x = pack_bf16x2(ov[8 * qq], ov[8 * qq + 1]);
              u.y = pack_bf16x2(ov[8 * qq + 2], ov[8 * qq + 3]);
              u.z = pack_bf16x2(ov[8 * qq + 4], ov[8 * qq + 5]);
              u.w = pack_bf16x2(ov[8 * qq + 6], ov[8 * qq + 7]);
              dst[qq] = u;
            }
          }
        }
        if (row_out && a.lse != nullptr) a.lse[orow] = (M + log2f(L)) * kLn2;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.ofree[t]);
      ++no;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int MODE>
cudaError_t launch_rows_dm(const AttnArgs& a, int num_sms, cudaStream_t stream) {
  PoolMaps m;
  cudaError_t e = encode_pool_maps(a, MODE != kRowsBlock, false, &m);
  if (e != cudaSuccess) return e;
  if (MODE == kRowsBlock) m.q = m.k;  // unused
  CUtensorMap tm_qb = m.k;            // the block queries in boxes of 64 rows
  if (MODE == kRowsBlock) {
    e = encode_3d_rows_sw128(&tm_qb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_block, D, a.n_heads,
                             a.bt.total_block_rows, 64, 64);
    if (e != cudaSuccess) return e;
  }
  constexpr int smem = RowsCfg<D>::kSmem;
  auto kern = rows_attn_kernel<D, MODE>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const long long rows = MODE == kRowsBlock ? a.bt.max_block_len : a.bt.max_seq_len;
  const long long pairs = (rows + 255) / 256;  // upper bound of a sequence's tile pairs
  for (int b0 = 0; b0 < a.bt.batch; b0 += kMaxSeqs) {
    const int n = a.bt.batch - b0 < kMaxSeqs ? a.bt.batch - b0 : kMaxSeqs;
    const long long units = static_cast<long long>(n) * a.n_heads * pairs;
    const int grid = static_cast<int>(units < num_sms ? units : num_sms);
    e = launch_pdl(kern, dim3(grid), kThreads, smem, 0, stream, m.q, tm_qb, m.k, m.v, a, b0, n);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_rows_d(const AttnArgs& a, int mode, int num_sms, cudaStream_t stream) {
  switch (mode) {
    case kRowsState:
      return launch_rows_dm<D, kRowsState>(a, num_sms, stream);
    case kRowsBlock:
      return launch_rows_dm<D, kRowsBlock>(a, num_sms, stream);
    case kRowsMerge:
      return launch_rows_dm<D, kRowsMerge>(a, num_sms, stream);
    case kRowsStatePre:
      return launch_rows_dm<D, kRowsStatePre>(a, num_sms, stream);
    case kRowsAdvOld:
      return launch_rows_dm<D, kRowsAdvOld>(a, num_sms, stream);
    default:
      return launch_rows_dm<D, kRowsAdvNew>(a, num_sms, stream);
  }
}

}  // namespace

cudaError_t launch_rows_attention(const AttnArgs& a, int mode, int num_sms, cudaStream_t stream) {
  if (a.bt.batch <= 0) return cudaSuccess;
  if (mode == kRowsBlock && a.bt.total_block_rows <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_rows_d<128>(a, mode, num_sms, stream) : launch_rows_d<64>(a, mode, num_sms, stream);
}

}  // namespace dllm
