// qkv_gemm.cu — fused RMSNorm + QKV projection + RoPE + single cache write
// (sm_103a), one kernel.
//
// Computes, for a set of token rows t (bf16 x_t), the normalised row
// x^_t = x_t / sqrt(mean(x_t^2) + eps) * g correctly rounded to bf16,
// y_t = W_qkv x^_t with fp32 accumulation, rotates the q and k parts (RoPE,
// rotate-half pairs (i, i + d/2) at the token's absolute position) and
// writes q, k, v once, as bf16, to their destinations: k, v into the paged
// pools through the block table, q into q_block (inner step) or q_pool
// (block boundary).  This is the Flash-Cache fusion of the Flash-dLLM
// write-up ("Flash-Cache: Fusing Projection, RoPE, and Cache Writes into One
// Kernel": projection and RoPE on chip, keys and values written straight
// into the cache in one HBM write) applied to the token-wise operators of
// LaCache §3.3.2, Eq. (1), with the RMSNorm in the same kernel.
//
// GB300 design.
//  * Swap-AB: the 128-row weight tiles are the tcgen05 M operand and the
//    (few) token rows are the N operand, so a 32-token inner step still fills
//    a 128 x 32 UMMA.
//  * The weight is stored tile-packed (every 128 x 64 box is 16 KB of
//    contiguous memory, the boxes of one weight tile in K order), so a CTA
//    streaming a tile's K range reads one contiguous run: measured on GB300,
//    96 CTAs then pull 100 MB at the same ~4.9 TB/s as 152, while with the
//    row-major layout (128-byte pieces of rows 8 KB apart) they reach ~3.9.
//  * A CTA that allocates TMEM runs alone on its SM, so the kernel is built
//    around one CTA per SM with a deep (~200 KB) TMA ring: warp 0 streams
//    units of K = 128 (one 32 KB weight load covering two boxes, two BN x 64
//    token boxes; 128-byte swizzle), warp 1 owns TMEM and issues
//    tcgen05.mma, warps 2-5 accumulate and write.
//  * Schedules.  Default: one CTA per (weight tile, token tile) over the full
//    K range: no cross-CTA reduction, so the kernel ends as soon as the last
//    weight bytes arrive.  When the weight tiles would occupy fewer than half
//    of the SMs (small models) the inner-step shapes (<= 64 token rows) are
//    scheduled stream-K instead: the (weight tile, k-unit) units are split
//    evenly over one CTA per SM; a weight tile that spans several CTAs is
//    finished by whichever contributor arrives last (fp32 partials in the
//    workspace, an atomic arrival counter; no CTA waits on another).
//  * fp32 accumulation on the CUDA cores ("promotion"): the tensor core sums
//    only the 128-element partial product of one unit (a chain of 8 MMAs)
//    into one of the TMEM buffers; the accumulator warps drain each finished
//    buffer into fp32 registers.  The tensor core's own long accumulation chains round
//    noticeably worse than fp32 round-to-nearest, and every bf16 value this
//    kernel stores is a cache entry that later steps reuse.  All 512 TMEM
//    columns serve as partial buffers, so the tensor core can run far ahead
//    while the accumulator warps finish a tile.
//  * RMSNorm inside the kernel.  A row's scale needs the whole row, and every
//    CTA multiplies all of its token rows, so each row is normalised once
//    for all CTAs: the accumulator warps claim rows through a counter in the
//    workspace (one atomic per claim), and a claiming warp reads the row,
//    forms its exact sum of squares and scale (float pairs), writes the
//    correctly rounded bf16 x^ row to the workspace and publishes it.  The
//    TMA producer waits until every row is published before it loads x^
//    tiles.  It waits only after all rows have been claimed (its own CTA's
//    warps claim until none is left) and a claimed row belongs to a running
//    warp that publishes it without waiting on anything, so the wait ends
//    whatever the number of resident CTAs.  The last CTA done with the
//    counters sets them back to zero.
//  * Programmatic dependent launch: the weight tiles (constants) of the first
//    ring stages are requested before waiting for the preceding kernel (which
//    may produce x), so the weight stream overlaps that kernel's tail.
#include "kernels.cuh"
#include "norm.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace dllm {
namespace {

constexpr int kThreads = 192;
constexpr int kAccThreads = kThreads - 64;  // warps 2-5
constexpr int kTileM = 128;                 // weight rows per tile (UMMA M)
constexpr int kTileK = 64;                  // K elements per TMA box (one 128-byte swizzle row)
constexpr int kBoxes = 2;                   // boxes per unit: a unit covers K = 128
constexpr int kUnitK = kTileK * kBoxes;
constexpr int kTileABytes = kTileM * kTileK * 2;
constexpr int kMinUnitsPerCta = 4;
constexpr int kWideMinTokens = 256;         // from here on the wide-tile kernel (qkv_wide.cu)
constexpr int kSmemLimit = 232448 - 4096;   // opt-in maximum less room for the static shared data

template <int BN>
struct GemmCfg;
template <>
struct GemmCfg<32> {
  static constexpr int kStages = 5;
  static constexpr bool kOwnRecv = true;  // stream-K: tile epilogues run while the ring is busy
};
template <>
struct GemmCfg<64> {
  static constexpr int kStages = 3;
  static constexpr bool kOwnRecv = true;
};
template <>
struct GemmCfg<128> {
  static constexpr int kStages = 3;
  static constexpr bool kOwnRecv = false;  // one tile per CTA: the drained ring holds the tile
};

template <int BN>
constexpr int tmem_bufs() {
  return 512 / BN;
}
template <int BN>
constexpr int stage_bytes() {
  return kBoxes * (kTileABytes + BN * kTileK * 2);
}
template <int BN>
constexpr int ring_bytes() {
  return GemmCfg<BN>::kStages * stage_bytes<BN>();
}
template <int BN>
constexpr int gemm_smem_bytes() {
  return ring_bytes<BN>() + (GemmCfg<BN>::kOwnRecv ? BN * kTileM * 4 : 0) + 1024;
}
static_assert(gemm_smem_bytes<32>() <= kSmemLimit && gemm_smem_bytes<64>() <= kSmemLimit &&
                  gemm_smem_bytes<128>() <= kSmemLimit,
              "ring too large");
static_assert(ring_bytes<128>() >= 128 * kTileM * 4, "the drained ring must hold a 128-column tile");

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Largest b in [0, batch) with cu[b] <= j.
__device__ __forceinline__ int find_seq(const int32_t* cu, int batch, int j) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= j)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Stream-K split of U units over G CTAs: CTA c owns [c*U/G, (c+1)*U/G).
__host__ __device__ __forceinline__ long long sk_begin(long long c, long long U, long long G) { return c * U / G; }
__host__ __device__ __forceinline__ int sk_cta_of(long long u, long long U, long long G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// Walk of a CTA's units: weight tile, k-unit, and where segments (runs of one
// tile) begin and end.  The producer, the MMA issuer and the accumulator
// warps all follow the same walk, advanced incrementally (no integer division
// inside the loops).
struct UnitWalk {
  int tile, kb, ps;  // weight tile, k-unit, position inside the segment
  int nkb, left;     // k-units per tile, units left after this one
  bool seg_end;
  __device__ __forceinline__ void init(long long u0, long long u1, int nkb_) {
    nkb = nkb_;
    tile = static_cast<int>(u0 / nkb);
    kb = static_cast<int>(u0 % nkb);
    ps = 0;
    left = static_cast<int>(u1 - u0) - 1;
    seg_end = left == 0 || kb == nkb - 1;
  }
  __device__ __forceinline__ int seg_kb0() const { return kb - ps; }
  __device__ __forceinline__ void next() {
    --left;
    if (++kb == nkb) {
      kb = 0;
      ++tile;
      ps = 0;
    } else {
      ++ps;
    }
    seg_end = left == 0 || kb == nkb - 1;
  }
};



template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const QkvArgs a) {
  constexpr int kStages = GemmCfg<BN>::kStages;
  constexpr int kTileBBytes = BN * kTileK * 2;
  constexpr int kStageBytes = stage_bytes<BN>();  // A box 0 | A box 1 | B box 0 | B box 1
  constexpr int kTmemBufs = tmem_bufs<BN>();
  constexpr uint32_t kTmemCols = kTmemBufs * BN;  // 512: the CTA is alone on its SM
  constexpr uint32_t kIdesc = umma_idesc_bf16(kTileM, BN);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float* recv = reinterpret_cast<float*>(smem + (GemmCfg<BN>::kOwnRecv ? ring_bytes<BN>() : 0));  // [BN][128]

  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[kTmemBufs], tempty_bar[kTmemBufs];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int last_sh;
  __shared__ int claim_sh[2];         // RMSNorm: the claimed row (slots alternate between rows)
  __shared__ float2 red_sh[2][kAccThreads / 32], scale_sh[2];
  __shared__ long long tok_kv[BN];  // element offset of (page, head 0, slot) in the pools, -1: no write
  __shared__ long long tok_q[BN];   // element offset of the q destination for head 0, -1: no write
  __shared__ int tok_pos[BN];       // absolute position (RoPE)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (a.d_model + kUnitK - 1) / kUnitK;  // a ragged last unit reads the packed zeros past d_model
  const int kbp = 2 * nkb;                            // packed boxes per weight tile
  const int n_wt = 3 * a.n_heads * a.head_dim / kTileM;
  const bool streamk = a.partials != nullptr;
  const int nt = streamk ? 0 : static_cast<int>(blockIdx.x);  // token tile (x: the tiles of one weight tile
                                                               // run side by side and share it in L2)
  const long long U = static_cast<long long>(n_wt) * nkb, G = gridDim.x;
  long long u0, u1;  // unit range of this CTA
  if (streamk) {
    u0 = sk_begin(blockIdx.x, U, G);
    u1 = sk_begin(blockIdx.x + 1, U, G);
  } else {
    u0 = static_cast<long long>(blockIdx.y) * nkb;
    u1 = u0 + nkb;
  }
  const int n_units = static_cast<int>(u1 - u0);
  const BatchArgs& bt = a.bt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < kTmemBufs; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kAccThreads / 32);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // Let the next kernel (the step's attention) start on the SMs this grid leaves
  // free: it streams what this kernel does not write while the weights stream.
  griddep_launch_dependents();

  if (warp == 0) {
    // ---- TMA producer.  Weight tiles of the first stages go out before the
    // dependency wait (weights are constants); x^ tiles only once every row
    // has been normalised and published.
    const int npre = n_units < kStages ? n_units : kStages;
    UnitWalk w;
    w.init(u0, u1, nkb);
    const uint64_t wpol = l2_evict_first_policy();  // each weight byte is read once per call
    if (lane == 0) {
      for (int i = 0; i < npre; ++i, w.next()) {
        mbar_arrive_expect_tx(&full_bar[i], kStageBytes);
        tma_load_2d_hint(smem + i * kStageBytes, &tm_w, &full_bar[i], 0, (w.tile * kbp + kBoxes * w.kb) * kTileM,
                         wpol);
      }
      griddep_wait();
      const uint64_t t0 = global_timer_ns();  // bounded wait for the x^ rows
      while (ld_acquire_gpu(a.norm_ctr + 1) < a.n_tok) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        __nanosleep(20);
      }
      fence_proxy_async_global();  // the rows written by other CTAs' threads, as seen by TMA
    }
    __syncwarp();
    named_barrier_arrive(2, 32 + kAccThreads);  // this CTA no longer reads the claim counters
    named_barrier(3, 32 + kAccThreads);         // this CTA's RMSNorm staging areas are free for x^ tiles
    if (lane == 0) {
      {
        UnitWalk wb;
        wb.init(u0, u1, nkb);
        for (int i = 0; i < npre; ++i, wb.next())
#pragma unroll
          for (int j = 0; j < kBoxes; ++j)
            tma_load_2d(smem + i * kStageBytes + kBoxes * kTileABytes + j * kTileBBytes, &tm_x, &full_bar[i],
                        wb.kb * kUnitK + j * kTileK, nt * BN);
      }
      int issued = npre;
      int s = npre % kStages;
      uint32_t ph = (npre / kStages) & 1;
      for (int i = npre; i < n_units; ++i, w.next()) {
        if (!mbar_wait(&empty_bar[s], ph ^ 1)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        uint8_t* sa = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        tma_load_2d_hint(sa, &tm_w, &full_bar[s], 0, (w.tile * kbp + kBoxes * w.kb) * kTileM, wpol);
#pragma unroll
        for (int j = 0; j < kBoxes; ++j)
          tma_load_2d(sa + kBoxes * kTileABytes + j * kTileBBytes, &tm_x, &full_bar[s], w.kb * kUnitK + j * kTileK,
                      nt * BN);
        ++issued;
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      // Drain: every issued load has landed before the CTA can retire.
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report_error(bt.err, kErrTimeout);
      // Tail: the MMA issuer's last releases of the ring (tcgen05.commit arrivals on
      // empty_bar, which nothing else waits for) have landed too.  No asynchronous
      // arrival may reach this CTA's shared memory after it exits: under programmatic
      // dependent launch the next kernel's CTA can start on this SM at once, with its
      // own barriers at the same offsets.
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        if (!mbar_wait(&empty_bar[i % kStages], (i / kStages) & 1)) report_error(bt.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer: unit i = round * kTmemBufs + buf goes to TMEM buffer buf.
      bool ok = true;
      int buf = kTmemBufs - 1, round = -1;
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_units && ok; ++i) {
        if (++buf == kTmemBufs) {
          buf = 0;
          ++round;
        }
        if (round >= 1 && !mbar_wait(&tempty_bar[buf], (round + 1) & 1)) {
          report_error(bt.err, kErrTimeout);
          ok = false;
          break;
        }
        if (!mbar_wait(&full_bar[s], ph)) {
          report_error(bt.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * kStageBytes), sb = sa + kBoxes * kTileABytes;
        const uint32_t d = tmem + static_cast<uint32_t>(buf * BN);
#pragma unroll
        for (int k = 0; k < kUnitK / 16; ++k) {
          const int j = k / (kTileK / 16), kk = k % (kTileK / 16);
          umma_bf16(d, umma_desc_sw128(sa + j * kTileABytes + kk * 32), umma_desc_sw128(sb + j * kTileBBytes + kk * 32),
                    kIdesc, k == 0 ? 0u : 1u);
        }
        umma_commit(&empty_bar[s]);
        umma_commit(&tfull_bar[buf]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok)  // let the accumulator warps finish (their waits see the phases they expect)
        for (int b = 0; b < kTmemBufs; ++b) umma_commit(&tfull_bar[b]);
    }
    __syncwarp();
  } else {
    // ---- accumulator warps (TMEM lane quarter = warp % 4)
    const int H = a.n_heads, d = a.head_dim, half = d >> 1;
    const int HD = H * d;
    // RMSNorm: the CTA's accumulator warps claim one row at a time until none
    // is left.  Until the producer loads x^ tiles, the x^ areas of ring
    // stages 0 and 1 are free: the row and the gain are staged there, each
    // thread in its own 16-byte slots (vectors at + 128 j), so the code is a
    // few short loops (this runs once per launch, from a cold instruction
    // cache).
    {
      const int at = threadIdx.x - 64;
      const uint4* xg = static_cast<const uint4*>(a.x);
      const uint4* gg = static_cast<const uint4*>(a.gain);
      uint4* xh = static_cast<uint4*>(a.xhat);
      const int nvec = a.d_model / 8;
      constexpr int kCap = kBoxes * kTileBBytes / 16;  // 16-byte vectors in one stage's x^ area
      uint4* rowbuf = reinterpret_cast<uint4*>(smem + kBoxes * kTileABytes);
      uint4* gainbuf = reinterpret_cast<uint4*>(smem + kStageBytes + kBoxes * kTileABytes);
      const bool staged = nvec <= kCap;  // the row fits: one load pass, the gain kept in shared memory
      if (staged)  // the gain is a layer constant: read before the dependency wait
        for (int v = at; v < nvec; v += kAccThreads) gainbuf[v] = __ldg(gg + v);
      // Iteration -1 runs the row code on zeros, with no loads, stores or
      // atomics, before the dependency wait: it brings the code into the
      // instruction cache while the preceding kernel finishes (the start
      // value comes through asm so that the compiler keeps one copy of the
      // loop body).
      int it0;
      asm volatile("mov.b32 %0, -1;" : "=r"(it0));
      for (int it = it0;; ++it) {
        const bool warm = it < 0;
        const int par = it & 1;  // the shared slots alternate between consecutive rows
        if (at == 0) claim_sh[par] = warm ? 0 : atomicAdd(a.norm_ctr, 1);
        named_barrier(1, kAccThreads);
        const int r = claim_sh[par];
        if (r >= a.n_tok) break;
        const uint4* xr = xg + static_cast<size_t>(r) * nvec;
        uint4* hr = xh + static_cast<size_t>(r) * nvec;
        float hi = 0.f, lo = 0.f;
        for (int c0 = 0; c0 < nvec; c0 += kCap) {  // exact sum of squares, a staged chunk at a time
          const int n = min(kCap, nvec - c0);
#pragma unroll 4
          for (int v = at; v < n; v += kAccThreads)
            rowbuf[v] = warm ? make_uint4(0, 0, 0, 0) : __ldg(xr + c0 + v);
#pragma unroll 1
          for (int v = at; v < n; v += kAccThreads) sumsq_pair_add(rowbuf[v], hi, lo);
        }
#pragma unroll 1
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
          pair_add(hi, lo, oh, ol);
        }
        if (lane == 0) red_sh[par][warp - 2] = make_float2(hi, lo);
        named_barrier(1, kAccThreads);
        if (at == 0) {  // the four warps' sums in a fixed order, then the scale
          float ss_hi = red_sh[par][0].x, ss_lo = red_sh[par][0].y;
#pragma unroll 1
          for (int q = 1; q < kAccThreads / 32; ++q) pair_add(ss_hi, ss_lo, red_sh[par][q].x, red_sh[par][q].y);
          two_sum(ss_hi, ss_lo, ss_hi, ss_lo);
          float y_hi, y_lo;
          rsqrt_pair(ss_hi, ss_lo, a.d_model, a.rms_eps, y_hi, y_lo);
          scale_sh[par] = make_float2(y_hi, y_lo);
          if (!warm) a.inv[r] = make_float2(y_hi, y_lo);
        }
        named_barrier(1, kAccThreads);
        const float2 y = scale_sh[par];
#pragma unroll 1
        for (int v = at; v < nvec; v += kAccThreads) {  // x^, correctly rounded
          const uint4 xv = staged ? rowbuf[v] : (warm ? make_uint4(0, 0, 0, 0) : __ldg(xr + v));
          const uint4 gvv = staged ? gainbuf[v] : __ldg(gg + v);
          const uint4 o = normalise8(xv, gvv, y.x, y.y);
          if (!warm) hr[v] = o;
        }
        fence_proxy_async_global();  // the row will be read by TMA
        named_barrier(1, kAccThreads);
        if (warm) {
          griddep_wait();  // from here on x may be read
          continue;
        }
        if (at == 0) red_release_gpu_add(a.norm_ctr + 1, 1);  // the row and its scale, then the count
      }
      // the staging areas are about to be written by TMA (async proxy)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_barrier_arrive(3, 32 + kAccThreads);
    }
    for (int c = threadIdx.x - 64; c < BN; c += kAccThreads) {  // resolve token columns
      long long kv = -1, qd = -1;
      int pos = 0;
      const int j = nt * BN + c;
      if (j < a.n_tok) {
        const int32_t* cu = a.mode == kModeBoundary ? bt.cu_seq : bt.cu_block;
        const int b = find_seq(cu, bt.batch, j);
        const int off = j - __ldg(cu + b);
        const int nb = __ldg(bt.seq_len + b), sb = __ldg(bt.block_start + b), lb = __ldg(bt.block_len + b);
        pos = a.mode == kModeBoundary ? off : sb + off;
        const bool shape_ok = nb >= 1 && nb <= bt.max_seq_len && lb >= 1 && lb <= bt.max_block_len && sb >= 0 &&
                              sb + lb <= nb && (a.mode == kModeBoundary ? off < nb : off < lb) && pos >= 0 &&
                              pos < nb && pos < a.rope_max_pos && pos / kPage < bt.max_pages;
        if (!shape_ok) {
          report_error(bt.err, kErrBadShape);
        } else {
          const int pg = __ldg(bt.block_table + static_cast<size_t>(b) * bt.max_pages + pos / kPage);
          if (pg < 0 || pg >= bt.num_pages) {
            report_error(bt.err, kErrBadPage);
          } else {
            kv = (static_cast<long long>(pg) * H * kPage + (pos % kPage)) * d;
            if (a.mode == kModeBlock)
              qd = static_cast<long long>(j) * H * d;
            else if (a.mode == kModeRows || pos < sb || pos >= sb + lb)
              qd = kv;  // queries are cached for the invariant rows (and the rows of a range) only
          }
        }
      }
      tok_kv[c] = kv;
      tok_q[c] = qd;
      tok_pos[c] = kv >= 0 ? pos : 0;  // a checked position (the RoPE table is read for every column)
    }
    // Once this CTA's producer has seen every row published (and its own
    // warps have stopped claiming), the CTA is done with the claim counters;
    // the last CTA to get there zeroes them for the next call.
    named_barrier(2, 32 + kAccThreads);
    if (threadIdx.x == 64) {
      const int n_cta = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
      if (atomicAdd(a.norm_ctr + 2, 1) == n_cta - 1) {
        a.norm_ctr[0] = 0;
        a.norm_ctr[1] = 0;
        a.norm_ctr[2] = 0;
      }
    }
    named_barrier(1, kAccThreads);

    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int ncols = min(BN, a.n_tok - nt * BN);
    __nv_bfloat16* kpool = static_cast<__nv_bfloat16*>(a.k_pool);
    __nv_bfloat16* vpool = static_cast<__nv_bfloat16*>(a.v_pool);
    __nv_bfloat16* qdst = static_cast<__nv_bfloat16*>(a.mode == kModeBlock ? a.q_block : a.q_pool);
    const int chunks_per_half = half / 8;  // 8 (d = 128) or 4 (d = 64)
    // Epilogue items: (token column c, 8-element chunk jc of the tile's low
    // halves).  A thread's items are the same for every tile, so with few
    // columns their RoPE factors are loaded once, here, off the tail.
    constexpr int kItems = BN * 8 / kAccThreads;
    constexpr bool kRopeRegs = BN <= 64;
    float4 rope_r[kRopeRegs ? kItems : 1][4];
    if constexpr (kRopeRegs) {
#pragma unroll
      for (int it = 0; it < kItems; ++it) {
        const int item = threadIdx.x - 64 + it * kAccThreads, c = item >> 3, jc = item & 7;
        const int t0 = (jc % chunks_per_half) * 8;
        const float4* cs =
            reinterpret_cast<const float4*>(a.rope + (static_cast<size_t>(tok_pos[c]) * half + t0) * 2);
#pragma unroll
        for (int e = 0; e < 4; ++e) rope_r[it][e] = __ldg(cs + e);
      }
    }
    float acc[BN];
#pragma unroll
    for (int c = 0; c < BN; ++c) acc[c] = 0.f;
    int buf = kTmemBufs - 1, round = -1;
    bool ok = true;  // after a timed-out wait the walk continues (same named barriers) without waiting
    UnitWalk w;
    w.init(u0, u1, nkb);
    for (int i = 0; i < n_units; ++i, w.next()) {
      if (++buf == kTmemBufs) {
        buf = 0;
        ++round;
      }
      if (ok && !mbar_wait(&tfull_bar[buf], round & 1)) {
        report_error(bt.err, kErrTimeout);
        ok = false;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) tmem_ld_add_32(lane_base + static_cast<uint32_t>(buf * BN + c0), acc + c0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
      if (!w.seg_end) continue;

      // ---- a segment (one weight tile's k-range of this CTA) is complete
      const int tile = w.tile;
      if (!(w.seg_kb0() == 0 && w.kb == nkb - 1)) {
        // Stream-K fixup: every contributor publishes its fp32 partial; the
        // last to arrive sums all of them in slot order (its own too, as
        // written), so the rounding does not depend on the arrival order.
        const int c_first = sk_cta_of(static_cast<long long>(tile) * nkb, U, G);
        const int c_last = sk_cta_of(static_cast<long long>(tile) * nkb + nkb - 1, U, G);
        const int n_other = c_last - c_first;
        const int slot = static_cast<int>(blockIdx.x) - c_first;
        float* slots = a.partials + static_cast<size_t>(tile) * a.max_contrib * kTileM * BN;
        float* mine = slots + static_cast<size_t>(slot) * kTileM * BN + static_cast<size_t>(row) * BN;
#pragma unroll
        for (int c = 0; c < BN; c += 4)
          *reinterpret_cast<float4*>(mine + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        named_barrier(1, kAccThreads);  // the CTA's partial rows are written ...
        if (threadIdx.x == 64) {
          __threadfence();  // ... and (cumulatively) visible GPU-wide before the arrival is counted
          last_sh = atomicAdd(a.counters + tile, 1) == n_other ? 1 : 0;
        }
        named_barrier(1, kAccThreads);
#pragma unroll
        for (int c = 0; c < BN; ++c) acc[c] = 0.f;
        if (!last_sh) continue;
        __threadfence();
        for (int sl = 0; sl <= n_other; ++sl) {
          const float* part = slots + static_cast<size_t>(sl) * kTileM * BN + static_cast<size_t>(row) * BN;
#pragma unroll
          for (int c = 0; c < BN; c += 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(part + c));
            acc[c] += v.x;
            acc[c + 1] += v.y;
            acc[c + 2] += v.z;
            acc[c + 3] += v.w;
          }
        }
        if (threadIdx.x == 64) a.counters[tile] = 0;  // ready for the next call
      }

      // ---- epilogue of one weight tile: rotate q/k, round to bf16, write 16-byte runs
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        recv[c * kTileM + row] = acc[c];
        acc[c] = 0.f;
      }
      named_barrier(1, kAccThreads);
      const int grow0 = tile * kTileM;
      const int which = grow0 / HD;  // 0: q, 1: k, 2: v
      const int head0 = (grow0 % HD) / d;
#pragma unroll
      for (int it = 0; it < (kRopeRegs ? kItems : 1); ++it) {
        for (int item = threadIdx.x - 64 + it * kAccThreads; item < ncols * 8;
             item += (kRopeRegs ? ncols * 8 : kAccThreads)) {
          const int c = item >> 3, jc = item & 7;
          const long long kv = tok_kv[c];
          if (kv < 0) continue;
          const int hit = jc / chunks_per_half, t0 = (jc % chunks_per_half) * 8;
          const int row_lo = hit * d + t0, row_hi = row_lo + half;
          float lo[8], hi[8];
          const float* r = recv + c * kTileM;
#pragma unroll
          for (int e = 0; e < 8; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(r + row_lo + e);
            const float4 h4 = *reinterpret_cast<const float4*>(r + row_hi + e);
            lo[e] = l4.x;
            lo[e + 1] = l4.y;
            lo[e + 2] = l4.z;
            lo[e + 3] = l4.w;
            hi[e] = h4.x;
            hi[e + 1] = h4.y;
            hi[e + 2] = h4.z;
            hi[e + 3] = h4.w;
          }
          const int head = head0 + hit;
          __nv_bfloat16* out;
          if (which == 2) {
            out = vpool + kv + static_cast<long long>(head) * kPage * d;
          } else {
            float4 cs[4];
            if constexpr (kRopeRegs) {
#pragma unroll
              for (int e = 0; e < 4; ++e) cs[e] = rope_r[it][e];
            } else {
              const float4* tab =
                  reinterpret_cast<const float4*>(a.rope + (static_cast<size_t>(tok_pos[c]) * half + t0) * 2);
#pragma unroll
              for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + e);
            }
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float4 v = cs[e / 2];  // (cos, sin) of t0+e and t0+e+1
              const float l0 = lo[e] * v.x - hi[e] * v.y, h0 = hi[e] * v.x + lo[e] * v.y;
              const float l1 = lo[e + 1] * v.z - hi[e + 1] * v.w, h1 = hi[e + 1] * v.z + lo[e + 1] * v.w;
              lo[e] = l0;
              hi[e] = h0;
              lo[e + 1] = l1;
              hi[e + 1] = h1;
            }
            if (which == 1) {
              out = kpool + kv + static_cast<long long>(head) * kPage * d;
            } else {
              const long long qd = tok_q[c];
              if (qd < 0) continue;
              out = qdst + qd + static_cast<long long>(head) * (a.mode == kModeBlock ? d : kPage * d);
            }
          }
          uint4 wl, wh;
          wl.x = pack_bf16x2(lo[0], lo[1]);
          wl.y = pack_bf16x2(lo[2], lo[3]);
          wl.z = pack_bf16x2(lo[4], lo[5]);
          wl.w = pack_bf16x2(lo[6], lo[7]);
          wh.x = pack_bf16x2(hi[0], hi[1]);
          wh.y = pack_bf16x2(hi[2], hi[3]);
          wh.z = pack_bf16x2(hi[4], hi[5]);
          wh.w = pack_bf16x2(hi[6], hi[7]);
          *reinterpret_cast<uint4*>(out + t0) = wl;
          *reinterpret_cast<uint4*>(out + t0 + half) = wh;
        }
      }
      named_barrier(1, kAccThreads);  // recv is free for the next tile
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN>
cudaError_t launch_bn(const void* w_packed, const QkvArgs& a, const QkvPlan& plan, cudaStream_t stream) {
  const int HD = a.n_heads * a.head_dim;
  CUtensorMap tm_w, tm_x;
  // the packed weight as rows of 64 columns; one load = the two boxes of a unit
  const uint64_t w_rows = static_cast<uint64_t>(3 * HD / kTileM) * qkv_boxes_per_tile(a.d_model) * kTileM;
  cudaError_t e = encode_2d_sw128(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_packed, kTileK, w_rows, kTileK,
                                  kBoxes * kTileM);
  if (e != cudaSuccess) return e;
  e = encode_2d_sw128(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.xhat, a.d_model, a.n_tok, kTileK, BN);
  if (e != cudaSuccess) return e;
  auto kern = qkv_gemm_kernel<BN>;
  constexpr int smem = gemm_smem_bytes<BN>();
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)  // all of the unified L1/shared storage as shared memory
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int n_wt = 3 * HD / kTileM;
  cfg.gridDim = plan.streamk ? dim3(plan.grid, 1, 1) : dim3((a.n_tok + BN - 1) / BN, n_wt, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, a);
}

}  // namespace

QkvPlan qkv_plan(int n_tok, int d_model, int n_heads, int head_dim, int num_sms) {
  QkvPlan p = {};
  const long long n_wt = 3LL * n_heads * head_dim / kTileM;
  const long long nkb = (d_model + kUnitK - 1) / kUnitK;
  p.inv_offset = kQkvCounterBytes;
  p.inv_bytes = align256(static_cast<size_t>(n_tok) * 8);
  p.xhat_offset = p.inv_offset + p.inv_bytes;
  p.xhat_bytes = align256(static_cast<size_t>(n_tok) * d_model * 2);
  p.part_offset = p.xhat_offset + p.xhat_bytes;
  if (n_tok >= kWideMinTokens) {  // tensor-bound: the persistent wide-tile kernel
    qkv_wide_schedule(n_tok, d_model, n_heads, head_dim, num_sms, &p);
    p.part_bytes = align256(p.part_bytes);
    p.total_bytes = p.part_offset + p.part_bytes;
    return p;
  }
  p.bn = n_tok <= 32 ? 32 : (n_tok <= 64 ? 64 : 128);
  p.streamk = p.bn <= 64 && 2 * n_wt <= num_sms && n_wt <= kQkvMaxTileCounters;
  if (p.streamk) {
    const long long U = n_wt * nkb;
    long long G = U / kMinUnitsPerCta;
    if (G > num_sms) G = num_sms;
    if (G < 1) G = 1;
    p.grid = static_cast<int>(G);
    int maxc = 1;
    for (long long t = 0; t < n_wt; ++t) {
      const int c = sk_cta_of(t * nkb + nkb - 1, U, G) - sk_cta_of(t * nkb, U, G) + 1;
      if (c > maxc) maxc = c;
    }
    p.max_contrib = maxc;
    p.part_bytes = align256(static_cast<size_t>(n_wt) * maxc * kTileM * p.bn * 4);
  }
  p.total_bytes = p.part_offset + p.part_bytes;
  return p;
}

cudaError_t launch_qkv_gemm(const void* w_packed, const QkvArgs& a, const QkvPlan& plan, cudaStream_t stream) {
  if (a.n_tok <= 0) return cudaSuccess;
  if (plan.wide) return launch_qkv_wide(w_packed, a, plan, stream);
  if (plan.bn == 32) return launch_bn<32>(w_packed, a, plan, stream);
  if (plan.bn == 64) return launch_bn<64>(w_packed, a, plan, stream);
  return launch_bn<128>(w_packed, a, plan, stream);
}

namespace {
// One thread per 16-byte chunk of the packed weight (zeros past d_model).
__global__ void qkv_pack_kernel(const uint4* __restrict__ w, uint4* __restrict__ packed, int rows, int d_model,
                                int kbp, long long n_chunks) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n_chunks) return;
  const int ch = static_cast<int>(idx & 7);
  const long long box_row = idx >> 3;  // ((t * kbp + kb) * 128 + r)
  const int r = static_cast<int>(box_row % kTileM);
  const long long tk = box_row / kTileM;
  const int kb = static_cast<int>(tk % kbp);
  const long long t = tk / kbp;
  const int col = kb * kTileK + ch * 8;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (col < d_model) v = __ldg(w + ((t * kTileM + r) * d_model + col) / 8);
  packed[idx] = v;
}
}  // namespace

cudaError_t launch_qkv_pack(const void* w, void* packed, int rows, int d_model, cudaStream_t stream) {
  const int kbp = qkv_boxes_per_tile(d_model);
  const long long n_chunks = static_cast<long long>(rows / kTileM) * kbp * kTileM * 8;
  if (n_chunks == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (n_chunks + threads - 1) / threads;
  qkv_pack_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(w), static_cast<uint4*>(packed), rows, d_model, kbp, n_chunks);
  return cudaGetLastError();
}

}  // namespace dllm
