// qkv_wide.cu — the fused RMSNorm + QKV projection + RoPE + single cache write
// (sm_103a) for many token rows: the tensor-bound shapes (an inner step of a
// large batch, every block boundary).
//
// Same computation as qkv_gemm.cu (x^ = RMSNorm(x) correctly rounded to bf16,
// y = W_qkv x^ with fp32 accumulation, RoPE of the q and k parts at absolute
// positions, one bf16 write of q, k, v to their destinations; the Flash-Cache
// fusion of the Flash-dLLM write-up, "Flash-Cache: Fusing Projection, RoPE,
// and Cache Writes into One Kernel", on the token-wise operators of LaCache
// §3.3.2, Eq. (1)), organised for throughput:
//  * Persistent CTAs, one per SM, walking output tiles of 128 weight rows
//    (tcgen05 M) x 256 token rows (tcgen05 N = 256: one MMA instruction does
//    twice the work of a 128-wide tile, which halves the issue and
//    synchronisation cost per flop).  Tiles are numbered weight tile fastest,
//    so the CTAs running at one time share token rows and keep the weight
//    (about 100 MB for an 8B-shaped layer) resident in the 129 MB L2.
//  * With many tiles per SM every CTA takes whole tiles (tile c, c + G, ...).
//    With few (an inner step of a few hundred rows: a handful of tiles per
//    SM or less) the (tile, K chunk) units are split evenly over the CTAs
//    (stream-K); a tile split over several CTAs is finished by whichever
//    contributor arrives last, which sums every contributor's fp32 partial in
//    slot order (the rounding does not depend on the arrival order).
//  * Warp 0 streams K in stages of 64 (16 KB of packed weight + 32 KB of x^)
//    into a 4-stage ring with TMA; warp 1 issues the MMAs; warps 4-11 hold
//    the accumulators (128 fp32 each a thread: the first warpgroup hands
//    registers to them with setmaxnreg, since at 12 warps a sub-partition's
//    16 K registers allow 168 a thread).  fp32 promotion as in qkv_gemm.cu: the tensor core
//    sums one K chunk of 128 products into one of two 256-column TMEM
//    buffers, and the accumulator warps add each finished chunk into fp32
//    registers (two warps per TMEM lane quadrant, 128 columns each), so the
//    MMAs of the next chunk run while a chunk is drained.
//  * Epilogue: a tile's 256 columns go out 32 at a time through one 16 KB
//    staging tile (fp32 [32 columns][128 rows]): RoPE pairs (i, i + d/2) sit
//    in different TMEM quadrants, and each output row (one token, one head)
//    is d contiguous bf16.
//  * RMSNorm: every token row is normalised once for all CTAs before any x^
//    tile is loaded; the accumulator warps claim rows through a counter in
//    the workspace, one row per warp, and publish each (release-ordered
//    count).  A claimed row belongs to a running warp that waits on nothing,
//    so the producer's wait for all rows ends whatever the residency.
#include "kernels.cuh"
#include "norm.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace dllm {
namespace {

// Warpgroup 0: warp 0 TMA, warp 1 MMA (warps 2-3 idle); warpgroups 1-2 (warps 4-11): the
// accumulators.  Launched at kLaunchRegs registers a thread; warpgroup 0 then gives
// registers up (kFewRegs) and warpgroups 1-2 take them (kManyRegs): 4 x 32 x kFewRegs +
// 8 x 32 x kManyRegs == 12 x 32 x kLaunchRegs, also per SM sub-partition (one warp of each
// warpgroup per sub-partition).
constexpr int kThreads = 384;
constexpr int kFirstAccWarp = 4;
constexpr int kAccWarps = 8;
constexpr int kLaunchRegs = 168;
constexpr int kFewRegs = 56;
constexpr int kManyRegs = 224;
static_assert(4 * kFewRegs + 8 * kManyRegs == 12 * kLaunchRegs, "register split must add up to the launch");
constexpr int kAcc = kAccWarps * 32;     // accumulator threads
constexpr int kTM = 128;                 // weight rows per tile (tcgen05 M)
constexpr int kTN = 256;                 // token rows per tile (tcgen05 N)
constexpr int kBK = 64;                  // K per ring stage: one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kABytes = kTM * kBK * 2;   // 16 KB of packed weight
constexpr int kBBytes = kTN * kBK * 2;   // 32 KB of x^
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kStagingCols = 32;         // epilogue: token columns per pass
constexpr int kStagingBytes = kStagingCols * kTM * 4;
constexpr int kDynSmem = kStages * kStageBytes + kStagingBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;      // two chunk buffers of kTN columns
constexpr int kColsPerThread = kTN / 2;  // two accumulator warps per lane quadrant
constexpr int kPartialFloats = kTM * kTN;
constexpr int kNormVec = 16;             // RMSNorm: 16-byte pieces of a row a lane holds (rows up to 4096 wide)

// Stream-K: CTA c owns units [c U / G, (c + 1) U / G); the CTA that owns unit u.
__host__ __device__ __forceinline__ long long wk_begin(long long c, long long U, long long G) { return c * U / G; }
__host__ __device__ __forceinline__ int wk_cta_of(long long u, long long U, long long G) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

// Tile order: the weight tiles go in bands of `band` tiles (the last band may be
// narrower); within a band, token tile by token tile, weight tile fastest.  The CTAs
// running at one time then share one band of the weight, which stays resident in L2
// while every token tile passes over it (with all weight tiles in one order, each wave
// of tiles touched the whole weight and the pool writes evicted it between waves).
__device__ __forceinline__ void tile_coords(int tile, int n_wt, int n_tt, int band, int& wt, int& tt) {
  const int full = n_wt / band;  // bands of `band` weight tiles
  const int in_full = full * band * n_tt;
  if (tile < in_full) {
    const int b = tile / (band * n_tt), r = tile % (band * n_tt);
    tt = r / band;
    wt = b * band + r % band;
  } else {
    const int rest = n_wt - full * band, r = tile - in_full;
    tt = r / rest;
    wt = full * band + r % rest;
  }
}

// The walk of a CTA's work: segments (one tile, a contiguous range of its K
// chunks), chunk by chunk.  The producer, the MMA issuer and the
// accumulator warps all follow the same walk.
struct SegWalk {
  long long U;       // units (tile, chunk) in all
  int G, c, nck, n_tiles;
  bool sk;           // stream-K (else whole tiles c, c + G, ...)
  long long sk_u, sk_hi;
  int tile, c0, c1, ch;
  int wt, tt;  // the tile's weight tile and token tile
  int n_wt, n_tt, band;
  bool ok;

  __device__ __forceinline__ void init(int cta, int grid, int n_chunks, int tiles, bool streamk, int wtiles,
                                       int wband) {
    n_wt = wtiles;
    n_tt = tiles / wtiles;
    band = wband;
    c = cta;
    G = grid;
    nck = n_chunks;
    n_tiles = tiles;
    sk = streamk;
    U = static_cast<long long>(tiles) * n_chunks;
    ok = false;
    if (sk) {
      sk_u = wk_begin(c, U, G);
      sk_hi = wk_begin(c + 1, U, G);
      tile = -1;
    } else {
      tile = c - G;
    }
    next_segment();
  }
  __device__ __forceinline__ void next_segment() {
    if (sk) {
      ok = sk_u < sk_hi;
      if (!ok) return;
      tile = static_cast<int>(sk_u / nck);
      c0 = static_cast<int>(sk_u % nck);
      const long long left = sk_hi - sk_u;
      c1 = left < nck - c0 ? c0 + static_cast<int>(left) : nck;
      sk_u += c1 - c0;
    } else {
      tile += G;
      ok = tile < n_tiles;
      c0 = 0;
      c1 = nck;
    }
    ch = c0;
    if (ok) tile_coords(tile, n_wt, n_tt, band, wt, tt);
  }
  __device__ __forceinline__ void next_chunk() {
    if (++ch == c1) next_segment();
  }
  __device__ __forceinline__ bool seg_last() const { return ch == c1 - 1; }
  __device__ __forceinline__ bool whole() const { return c0 == 0 && c1 == nck; }
};

// The token columns of token tile tt: destination of k and v in the pools,
// of q (q_block in an inner step, q_pool at a boundary for the rows of U),
// and the absolute position (RoPE).  One column per accumulator thread.
__device__ __forceinline__ void resolve_columns(const QkvArgs& a, int tt, int at, long long* tok_kv, long long* tok_q,
                                                int* tok_pos) {
  const BatchArgs& bt = a.bt;
  const int d = a.head_dim, H = a.n_heads;
  long long kv = -1, qd = -1;
  int pos = 0;
  const int j = tt * kTN + at;
  if (j < a.n_tok) {
    const int32_t* cu = a.mode == kModeBoundary ? bt.cu_seq : bt.cu_block;
    int lo = 0, hi = bt.batch - 1;  // the sequence of token j: the largest b with cu[b] <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(cu + mid) <= j)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int b = lo;
    const int off = j - __ldg(cu + b);
    const int nb = __ldg(bt.seq_len + b), sb = __ldg(bt.block_start + b), lb = __ldg(bt.block_len + b);
    pos = a.mode == kModeBoundary ? off : sb + off;
    const bool shape_ok = nb >= 1 && nb <= bt.max_seq_len && lb >= 1 && lb <= bt.max_block_len && sb >= 0 &&
                          sb + lb <= nb && (a.mode == kModeBoundary ? off < nb : off < lb) && pos >= 0 && pos < nb &&
                          pos < a.rope_max_pos && pos / kPage < bt.max_pages;
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
  tok_kv[at] = kv;
  tok_q[at] = qd;
  tok_pos[at] = kv >= 0 ? pos : 0;  // a checked position (the RoPE table is read for every column)
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_wide_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const QkvArgs a, int n_wt, int band, int n_tiles, int streamk) {
  constexpr uint32_t kIdesc = umma_idesc_bf16(kTM, kTN);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float* staging = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [kStagingCols][kTM]

  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int last_sh;
  __shared__ long long tok_kv[kTN];
  __shared__ long long tok_q[kTN];
  __shared__ int tok_pos[kTN];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BatchArgs& bt = a.bt;
  const int kbp = 2 * ((a.d_model + 127) / 128);  // packed 64-column boxes per weight tile (zeros past d_model)
  const int nck = kbp / 2;                        // K chunks of 128
  const int G = static_cast<int>(gridDim.x);
  const bool sk = streamk != 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], kAccWarps);
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
  griddep_launch_dependents();

  if (warp < kFirstAccWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFewRegs));
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      // Weight halves of the first stages go out before the dependency wait (the
      // weight is a layer constant); x^ tiles only once every row is published.
      int npre = 0;
      if (lane == 0) {
        SegWalk w;
        w.init(blockIdx.x, G, nck, n_tiles, sk, n_wt, band);
        for (int k = 0; k < kStages / 2 && w.ok; ++k, w.next_chunk())
          for (int hb = 0; hb < 2; ++hb, ++npre) {
            mbar_arrive_expect_tx(&full_bar[npre], kStageBytes);
            tma_load_2d(smem + npre * kStageBytes, &tm_w, &full_bar[npre], 0,
                        (w.wt * kbp + 2 * w.ch + hb) * kTM);
          }
        griddep_wait();
        const uint64_t t0 = global_timer_ns();  // bounded wait for the x^ rows
        while (ld_acquire_gpu(a.norm_ctr + 1) < a.n_tok) {
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            report_error(bt.err, kErrTimeout);
            break;
          }
          __nanosleep(64);
        }
        fence_proxy_async_global();  // the rows written by other CTAs' threads, as seen by TMA
      }
      __syncwarp();
      named_barrier_arrive(2, 32 + kAcc);  // this CTA's producer no longer reads the claim counters
      if (lane == 0) {
        SegWalk w;
        w.init(blockIdx.x, G, nck, n_tiles, sk, n_wt, band);
        int q = 0;
        bool ok = true;
        for (; w.ok && ok; w.next_chunk()) {
          const int wt = w.wt, tt = w.tt;
          for (int hb = 0; hb < 2; ++hb, ++q) {
            const int s = q % kStages;
            uint8_t* st = smem + s * kStageBytes;
            if (q >= npre) {
              if (q >= kStages && !mbar_wait(&empty_bar[s], ((q / kStages) - 1) & 1)) {
                report_error(bt.err, kErrTimeout);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
              tma_load_2d(st, &tm_w, &full_bar[s], 0, (wt * kbp + 2 * w.ch + hb) * kTM);
            }
            tma_load_2d(st + kABytes, &tm_x, &full_bar[s], (2 * w.ch + hb) * kBK, tt * kTN);
          }
        }
        // Drain: every issued load has landed, and the MMA issuer's last releases of
        // the ring (tcgen05.commit arrivals nothing else waits for) have arrived, before
        // the CTA can exit (the next kernel's CTA may start on this SM at once).
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report_error(bt.err, kErrTimeout);
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&empty_bar[i % kStages], (i / kStages) & 1)) report_error(bt.err, kErrTimeout);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // Chunk n (K = 128: two ring stages) goes to TMEM buffer n % 2.
      if (lane == 0) {
        SegWalk w;
        w.init(blockIdx.x, G, nck, n_tiles, sk, n_wt, band);
        int q = 0, nc = 0;
        bool ok = true;
        for (; w.ok && ok; w.next_chunk(), ++nc) {
          const int b = nc & 1;
          if (nc >= 2 && !mbar_wait(&tempty_bar[b], ((nc >> 1) - 1) & 1)) {
            report_error(bt.err, kErrTimeout);
            ok = false;
            break;
          }
          const uint32_t d = tmem + static_cast<uint32_t>(b * kTN);
          for (int hb = 0; hb < 2; ++hb, ++q) {
            const int s = q % kStages;
            if (!mbar_wait(&full_bar[s], (q / kStages) & 1)) {
              report_error(bt.err, kErrTimeout);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kStageBytes), sb = sa + kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16(d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), kIdesc,
                        (hb > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&empty_bar[s]);
          }
          if (!ok) break;
          umma_commit(&tfull_bar[b]);
        }
        if (!ok)  // let the accumulator warps finish
          for (int b = 0; b < 2; ++b) umma_commit(&tfull_bar[b]);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kManyRegs));
    // ------------------------------------------------------------ accumulator warps
    const int ai = warp - kFirstAccWarp;     // 0..7
    const int quad = warp & 3;               // the TMEM lane quadrant this warp may read
    const int half = ai >> 2;                // the column half of a chunk buffer it drains
    const int at = threadIdx.x - 32 * kFirstAccWarp;  // 0..255
    const int row = quad * 32 + lane;        // weight row of the tile (TMEM lane)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int d = a.head_dim, H = a.n_heads, HD = H * d, half_d = d >> 1;

    // ---- RMSNorm: the warps of every CTA claim token rows, one row per warp.
    {
      const uint4* xg = static_cast<const uint4*>(a.x);
      const uint4* gg = static_cast<const uint4*>(a.gain);
      uint4* xh = static_cast<uint4*>(a.xhat);
      const int nvec = a.d_model / 8;
      griddep_wait();  // x may come from the preceding kernel
      for (;;) {
        int r = 0;
        if (lane == 0) r = atomicAdd(a.norm_ctr, 1);
        r = __shfl_sync(0xffffffffu, r, 0);
        if (r >= a.n_tok) break;
        const uint4* xr = xg + static_cast<size_t>(r) * nvec;
        uint4* hr = xh + static_cast<size_t>(r) * nvec;
        float hi = 0.f, lo = 0.f;  // exact sum of squares as a float pair
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) sumsq_pair_add(__ldg(xr + v), hi, lo);
#pragma unroll 1
        for (int o = 16; o > 0; o >>= 1) {
          const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
          pair_add(hi, lo, oh, ol);
        }
        float y_hi = 0.f, y_lo = 0.f;
        if (lane == 0) {  // lane 0's sum and scale are the row's
          two_sum(hi, lo, hi, lo);
          rsqrt_pair(hi, lo, a.d_model, a.rms_eps, y_hi, y_lo);
          a.inv[r] = make_float2(y_hi, y_lo);
        }
        y_hi = __shfl_sync(0xffffffffu, y_hi, 0);
        y_lo = __shfl_sync(0xffffffffu, y_lo, 0);
#pragma unroll 4
        for (int v = lane; v < nvec; v += 32) hr[v] = normalise8(__ldg(xr + v), __ldg(gg + v), y_hi, y_lo);
        fence_proxy_async_global();  // the row will be read by TMA
        __syncwarp();
        if (lane == 0) red_release_gpu_add(a.norm_ctr + 1, 1);  // the row and its scale, then the count
      }
    }
    // Once this CTA's producer has seen every row published (and its own warps have
    // stopped claiming), the CTA is done with the claim counters; the last CTA to get
    // there sets them back to zero for the next call.
    named_barrier(2, 32 + kAcc);
    if (at == 0 && atomicAdd(a.norm_ctr + 2, 1) == G - 1) {
      a.norm_ctr[0] = 0;
      a.norm_ctr[1] = 0;
      a.norm_ctr[2] = 0;
    }

    __nv_bfloat16* kpool = static_cast<__nv_bfloat16*>(a.k_pool);
    __nv_bfloat16* vpool = static_cast<__nv_bfloat16*>(a.v_pool);
    __nv_bfloat16* qdst = static_cast<__nv_bfloat16*>(a.mode == kModeBlock ? a.q_block : a.q_pool);
    const int chunks_per_half = half_d / 8;  // 8 (d = 128) or 4 (d = 64)
    float acc[kColsPerThread];
#pragma unroll
    for (int c = 0; c < kColsPerThread; ++c) acc[c] = 0.f;
    int cur_tt = -1;  // the token tile tok_* describe
    bool ok = true;   // after a timed-out wait the walk goes on (same barriers) without waiting
    SegWalk w;
    w.init(blockIdx.x, G, nck, n_tiles, sk, n_wt, band);
    for (int nc = 0; w.ok; w.next_chunk(), ++nc) {
      const int b = nc & 1;
      if (ok && !mbar_wait(&tfull_bar[b], (nc >> 1) & 1)) {
        report_error(bt.err, kErrTimeout);
        ok = false;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < kColsPerThread; c0 += 64)
        tmem_ld_add_64(lane_base + static_cast<uint32_t>(b * kTN + half * kColsPerThread + c0), acc + c0);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[b]);
      if (!w.seg_last()) continue;

      // ---- a segment (one tile's chunks of this CTA) is complete
      const int tile = w.tile;
      if (!w.whole()) {
        // Stream-K: every contributor publishes its fp32 partial; the last to arrive
        // sums all of them in slot order (its own too, as written).
        const long long u0 = static_cast<long long>(tile) * nck;
        const int c_first = wk_cta_of(u0, w.U, G), c_last = wk_cta_of(u0 + nck - 1, w.U, G);
        const int n_other = c_last - c_first;
        const int slot = static_cast<int>(blockIdx.x) - c_first;
        float4* mine = reinterpret_cast<float4*>(a.partials +
                                                 (static_cast<size_t>(tile) * a.max_contrib + slot) * kPartialFloats);
#pragma unroll
        for (int g = 0; g < kColsPerThread / 4; ++g)
          mine[g * kAcc + at] = make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2], acc[4 * g + 3]);
        named_barrier(1, kAcc);  // the CTA's partial is written ...
        if (at == 0) {
          __threadfence();  // ... and (cumulatively) visible GPU-wide before the arrival is counted
          last_sh = atomicAdd(a.counters + tile, 1) == n_other ? 1 : 0;
        }
        named_barrier(1, kAcc);
#pragma unroll
        for (int c = 0; c < kColsPerThread; ++c) acc[c] = 0.f;
        if (!last_sh) continue;
        __threadfence();
        for (int sl = 0; sl <= n_other; ++sl) {
          const float4* part = reinterpret_cast<const float4*>(
              a.partials + (static_cast<size_t>(tile) * a.max_contrib + sl) * kPartialFloats);
#pragma unroll
          for (int g = 0; g < kColsPerThread / 4; ++g) {
            const float4 v = __ldcg(part + g * kAcc + at);
            acc[4 * g] += v.x;
            acc[4 * g + 1] += v.y;
            acc[4 * g + 2] += v.z;
            acc[4 * g + 3] += v.w;
          }
        }
        if (at == 0) a.counters[tile] = 0;  // ready for the next call
      }

      // ---- epilogue of the tile: rotate q/k, round to bf16, write 16-byte runs
      const int wt = w.wt, tt = w.tt;
      if (tt != cur_tt) {
        named_barrier(1, kAcc);  // the previous tile's columns are no longer read
        resolve_columns(a, tt, at, tok_kv, tok_q, tok_pos);
        named_barrier(1, kAcc);
        cur_tt = tt;
      }
      const int grow0 = wt * kTM;
      const int which = grow0 / HD;  // 0: q, 1: k, 2: v
      const int head0 = (grow0 % HD) / d;
      constexpr int kPassesPerHalf = kColsPerThread / kStagingCols;
#pragma unroll
      for (int pass = 0; pass < (kTN / kStagingCols); ++pass) {
        const int ph = pass / kPassesPerHalf, pc = pass % kPassesPerHalf;
        if (half == ph) {
#pragma unroll
          for (int i = 0; i < kStagingCols; ++i) staging[i * kTM + row] = acc[pc * kStagingCols + i];
        }
        const int c = at >> 3, jc = at & 7;  // column of the pass, 8-element chunk of the tile's low halves
        const int col = ph * kColsPerThread + pc * kStagingCols + c;
        const int hit = jc / chunks_per_half, t0 = (jc % chunks_per_half) * 8;
        // the (cos, sin) of this thread's 8 pairs depend on the column's position only: loaded
        // before the barrier, so that their latency overlaps it
        float4 rope[4];
        if (which != 2) {
          const float4* tab =
              reinterpret_cast<const float4*>(a.rope + (static_cast<size_t>(tok_pos[col]) * half_d + t0) * 2);
#pragma unroll
          for (int e = 0; e < 4; ++e) rope[e] = __ldg(tab + e);
        }
        named_barrier(1, kAcc);
        {
          const long long kv = tok_kv[col];
          if (kv >= 0) {
            const int row_lo = hit * d + t0, row_hi = row_lo + half_d;
            const float* r = staging + c * kTM;
            float lo[8], hi[8];
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
            __nv_bfloat16* out = nullptr;
            if (which == 2) {
              out = vpool + kv + static_cast<long long>(head) * kPage * d;
            } else {
#pragma unroll
              for (int e = 0; e < 8; e += 2) {
                const float4 v = rope[e / 2];  // (cos, sin) of t0+e and t0+e+1
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
                const long long qd = tok_q[col];
                if (qd >= 0) out = qdst + qd + static_cast<long long>(head) * (a.mode == kModeBlock ? d : kPage * d);
              }
            }
            if (out != nullptr) {
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
              *reinterpret_cast<uint4*>(out + t0 + half_d) = wh;
            }
          }
        }
        named_barrier(1, kAcc);  // the staging tile is free for the next pass
      }
#pragma unroll
      for (int c = 0; c < kColsPerThread; ++c) acc[c] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace dllm

namespace dllm {

// The schedule of the wide kernel: whole tiles per CTA when every SM gets at
// least four of them (or when there are more tiles than the workspace has
// arrival counters), else stream-K over (tile, K chunk) units.
void qkv_wide_schedule(int n_tok, int d_model, int n_heads, int head_dim, int num_sms, QkvPlan* p) {
  const long long n_wt = 3LL * n_heads * head_dim / kTM;
  const long long n_tt = (n_tok + kTN - 1) / kTN;
  const long long n_tiles = n_wt * n_tt;
  const long long nck = (d_model + 127) / 128;
  p->wide = true;
  p->bn = kTN;
  p->n_tiles = static_cast<int>(n_tiles);
  p->streamk = n_tiles < 4LL * num_sms && n_tiles <= kQkvMaxTileCounters;
  p->max_contrib = 0;
  p->part_bytes = 0;
  if (p->streamk) {
    const long long U = n_tiles * nck;
    const long long G = U < num_sms ? U : num_sms;
    p->grid = static_cast<int>(G);
    int maxc = 1;
    for (long long t = 0; t < n_tiles; ++t) {
      const int c = wk_cta_of(t * nck + nck - 1, U, G) - wk_cta_of(t * nck, U, G) + 1;
      if (c > maxc) maxc = c;
    }
    p->max_contrib = maxc;
    p->part_bytes = static_cast<size_t>(n_tiles) * maxc * kPartialFloats * 4;
  } else {
    p->grid = static_cast<int>(n_tiles < num_sms ? n_tiles : num_sms);
  }
}

cudaError_t launch_qkv_wide(const void* w_packed, const QkvArgs& a, const QkvPlan& plan, cudaStream_t stream) {
  const int HD = a.n_heads * a.head_dim;
  const int n_wt = 3 * HD / kTM;
  CUtensorMap tm_w, tm_x;
  // the packed weight as rows of 64 columns, one 128 x 64 box (16 KB) per load
  const uint64_t w_rows = static_cast<uint64_t>(n_wt) * qkv_boxes_per_tile(a.d_model) * kTM;
  cudaError_t e = encode_2d_sw128(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_packed, kBK, w_rows, kBK, kTM);
  if (e != cudaSuccess) return e;
  e = encode_2d_sw128(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.xhat, a.d_model, a.n_tok, kBK, kTN);
  if (e != cudaSuccess) return e;
  // The register split inside the kernel assumes it was built at kLaunchRegs registers a
  // thread: with any other count its setmaxnreg.inc could not be satisfied, so refuse.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, qkv_wide_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(qkv_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  if (e == cudaSuccess)  // all of the unified L1/shared storage as shared memory
    e = cudaFuncSetAttribute(qkv_wide_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // weight band: about 48 MB of weight tiles (a third of L2), at least one tile
  const long long tile_bytes = static_cast<long long>(kTM) * qkv_boxes_per_tile(a.d_model) * kBK * 2;
  int band = static_cast<int>((48LL << 20) / tile_bytes);
  band = band < 1 ? 1 : (band > n_wt ? n_wt : band);
  return cudaLaunchKernelEx(&cfg, qkv_wide_kernel, tm_w, tm_x, a, n_wt, band, plan.n_tiles, plan.streamk ? 1 : 0);
}

}  // namespace dllm
