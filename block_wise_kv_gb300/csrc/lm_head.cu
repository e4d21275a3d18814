// lm_head.cu — the block-only epilogue after the layer stack (sm_103a): only
// the current block's rows go through the final RMSNorm, the LM head and the
// softmax over the vocabulary ("LaCache: Exact Caching and Precision-Adaptive
// Inference for Diffusion Large Language Models", §3.4: at the sampling stage
// the output is cut to the tokens of the current generation block; Fast-dLLM
// Block-wise DualCache, "Block-wise Generation": the inner step's logits are
// those of the block).
//
// Three kernels, chained by programmatic dependent launch:
//  * lm_gather_norm_kernel   one warp per block row: the row is read from the
//    full hidden states through the batch layout (row cu_seq[b] + s_b + i:
//    the truncation to the block), normalised (x^ = RMSNorm(h), correctly
//    rounded to bf16 as in the projection) into the workspace.
//  * lm_head_kernel          logits = x^ W_lm^T on the 5th-generation tensor
//    cores: persistent CTAs walking tiles of 128 rows (tcgen05 M) x 256
//    vocabulary entries (N = 256), vocabulary tiles in bands that stay
//    resident in L2 while every row tile passes over them.  Warp 0 streams
//    K in stages of 64 (16 KB of x^ + 32 KB of W_lm) into a 4-stage ring;
//    warp 1 issues the MMAs into two 256-column TMEM chunk buffers; warps
//    4-11 add each finished K chunk of 128 into fp32 registers (a thread
//    holds one row and 128 vocabulary entries) and, at the end of a tile,
//    reduce their 128 logits to (max, sum of exp(logit - max), first
//    argmax): one partial per (row, half tile), written to the workspace;
//    the logits themselves are written (bf16) only when asked for.
//  * lm_combine_kernel       one warp per row: the partials in vocabulary
//    order, merged exactly (the online-softmax merge of LaCache §3.3.3), into
//    L = log-sum-exp, the argmax (the lowest index among equal maxima) and
//    its probability exp(max - L).
#include <math.h>

#include "kernels.cuh"
#include "norm.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace dllm {
namespace {

constexpr int kThreads = 384;
constexpr int kFirstAccWarp = 4;
constexpr int kAccWarps = 8;
constexpr int kLaunchRegs = 168;
constexpr int kFewRegs = 56;
constexpr int kManyRegs = 224;
static_assert(4 * kFewRegs + 8 * kManyRegs == 12 * kLaunchRegs, "register split must add up to the launch");
constexpr int kTM = 128;                 // rows per tile (tcgen05 M)
constexpr int kTN = 256;                 // vocabulary entries per tile (tcgen05 N)
constexpr int kBK = 64;                  // K per ring stage
constexpr int kStages = 4;
constexpr int kABytes = kTM * kBK * 2;   // 16 KB of x^
constexpr int kBBytes = kTN * kBK * 2;   // 32 KB of W_lm
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kDynSmem = kStages * kStageBytes + 1024;
constexpr uint32_t kTmemCols = 512;      // two chunk buffers of kTN columns
constexpr int kColsPerThread = kTN / 2;

// ------------------------------------------------------------ gather + RMSNorm
// Block row j (packed by cu_block) of sequence b is row cu_seq[b] + s_b + (j - cu_block[b]) of
// the full hidden states; its normalised bf16 row goes to xhat[j].
__global__ void __launch_bounds__(256) lm_gather_norm_kernel(const LmArgs a) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  griddep_wait();  // h may come from the preceding kernel
  griddep_launch_dependents();
  const BatchArgs& bt = a.bt;
  const int j = warp;
  if (j >= a.n_rows) return;
  int lo = 0, hi = bt.batch - 1;  // the sequence of block row j: the largest b with cu_block[b] <= j
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(bt.cu_block + mid) <= j)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int b = lo, off = j - __ldg(bt.cu_block + b);
  const int nb = __ldg(bt.seq_len + b), sb = __ldg(bt.block_start + b), lb = __ldg(bt.block_len + b);
  const int cus = __ldg(bt.cu_seq + b);
  const int nvec = a.d_model / 8;
  uint4* xr = static_cast<uint4*>(a.xhat) + static_cast<size_t>(j) * nvec;
  const bool ok = nb >= 1 && nb <= bt.max_seq_len && lb >= 1 && lb <= bt.max_block_len && sb >= 0 && sb + lb <= nb &&
                  off >= 0 && off < lb && cus >= 0 && cus + nb <= bt.total_seq_rows;
  if (!ok) {
    if (lane == 0) report_error(bt.err, kErrBadShape);
    for (int v = lane; v < nvec; v += 32) xr[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* hr = static_cast<const uint4*>(a.h) + static_cast<size_t>(cus + sb + off) * nvec;
  const uint4* gg = static_cast<const uint4*>(a.gain);
  float shi = 0.f, slo = 0.f;  // exact sum of squares as a float pair
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) sumsq_pair_add(__ldg(hr + v), shi, slo);
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, shi, o), ol = __shfl_xor_sync(0xffffffffu, slo, o);
    pair_add(shi, slo, oh, ol);
  }
  float y_hi = 0.f, y_lo = 0.f;
  if (lane == 0) {  // lane 0's sum and scale are the row's
    two_sum(shi, slo, shi, slo);
    rsqrt_pair(shi, slo, a.d_model, a.rms_eps, y_hi, y_lo);
  }
  y_hi = __shfl_sync(0xffffffffu, y_hi, 0);
  y_lo = __shfl_sync(0xffffffffu, y_lo, 0);
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) xr[v] = normalise8(__ldg(hr + v), __ldg(gg + v), y_hi, y_lo);
}

// Tile order: vocabulary tiles in bands of `band` (the last may be narrower); within a band,
// row tile by row tile, vocabulary tile fastest.
__device__ __forceinline__ void lm_tile_coords(int tile, int n_vt, int n_tt, int band, int& vt, int& tt) {
  const int full = n_vt / band;
  const int in_full = full * band * n_tt;
  if (tile < in_full) {
    const int bi = tile / (band * n_tt), r = tile % (band * n_tt);
    tt = r / band;
    vt = bi * band + r % band;
  } else {
    const int rest = n_vt - full * band, r = tile - in_full;
    tt = r / rest;
    vt = full * band + r % rest;
  }
}

// ------------------------------------------------------------ LM head + softmax partials
__global__ void __launch_bounds__(kThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                   const LmArgs a, int n_vt, int n_tt, int band) {
  constexpr uint32_t kIdesc = umma_idesc_bf16(kTM, kTN);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nck = a.d_model / 128;  // K chunks of 128 (d_model is a multiple of 128)
  const int G = static_cast<int>(gridDim.x);
  const int n_tiles = n_vt * n_tt;

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
      if (lane == 0) {
        griddep_wait();  // x^ comes from the preceding kernel
        int q = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += G) {
          int vt, tt;
          lm_tile_coords(tile, n_vt, n_tt, band, vt, tt);
          for (int kb = 0; kb < 2 * nck; ++kb, ++q) {
            const int s = q % kStages;
            if (q >= kStages && !mbar_wait(&empty_bar[s], ((q / kStages) - 1) & 1)) {
              report_error(a.bt.err, kErrTimeout);
              ok = false;
              break;
            }
            uint8_t* st = smem + s * kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
            tma_load_2d(st, &tm_x, &full_bar[s], kb * kBK, tt * kTM);            // rows past n_rows read 0
            tma_load_2d(st + kABytes, &tm_w, &full_bar[s], kb * kBK, vt * kTN);  // entries past vocab read 0
          }
        }
        // Drain: every issued load has landed and the MMA issuer's last releases have arrived.
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report_error(a.bt.err, kErrTimeout);
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&empty_bar[i % kStages], (i / kStages) & 1)) report_error(a.bt.err, kErrTimeout);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        int q = 0, nc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += G) {
          for (int ck = 0; ck < nck && ok; ++ck, ++nc) {
            const int b = nc & 1;
            if (nc >= 2 && !mbar_wait(&tempty_bar[b], ((nc >> 1) - 1) & 1)) {
              report_error(a.bt.err, kErrTimeout);
              ok = false;
              break;
            }
            const uint32_t d = tmem + static_cast<uint32_t>(b * kTN);
            for (int hb = 0; hb < 2; ++hb, ++q) {
              const int s = q % kStages;
              if (!mbar_wait(&full_bar[s], (q / kStages) & 1)) {
                report_error(a.bt.err, kErrTimeout);
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
        }
        if (!ok)  // let the accumulator warps finish
          for (int b = 0; b < 2; ++b) umma_commit(&tfull_bar[b]);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kManyRegs));
    // ------------------------------------------------------------ accumulator warps
    const int ai = warp - kFirstAccWarp;  // 0..7
    const int quad = warp & 3;            // the TMEM lane quadrant this warp may read
    const int half = ai >> 2;             // the 128 vocabulary entries of a tile it holds
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    __nv_bfloat16* logits = static_cast<__nv_bfloat16*>(a.logits);
    float acc[kColsPerThread];
#pragma unroll
    for (int c = 0; c < kColsPerThread; ++c) acc[c] = 0.f;
    bool ok = true;
    int nc = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += G) {
      int vt, tt;
      lm_tile_coords(tile, n_vt, n_tt, band, vt, tt);
      for (int ck = 0; ck < nck; ++ck, ++nc) {
        const int b = nc & 1;
        if (ok && !mbar_wait(&tfull_bar[b], (nc >> 1) & 1)) {
          report_error(a.bt.err, kErrTimeout);
          ok = false;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kColsPerThread; c0 += 64)
          tmem_ld_add_64(lane_base + static_cast<uint32_t>(b * kTN + half * kColsPerThread + c0), acc + c0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
      }
      // ---- the tile is complete: this thread's row and 128 vocabulary entries
      const int row = tt * kTM + quad * 32 + lane;
      const int v0 = vt * kTN + half * kColsPerThread;
      const int nv = min(kColsPerThread, a.vocab - v0);  // entries of this half that exist (>= 1)
      if (row < a.n_rows && nv <= 0) {  // a half tile past the vocabulary: an empty partial
        const size_t pi = static_cast<size_t>(2 * vt + half) * a.n_rows + row;
        a.pmax[pi] = -INFINITY;
        a.psum[pi] = 0.f;
        a.parg[pi] = 0x7fffffff;
      } else if (row < a.n_rows) {
        if (logits != nullptr && nv == kColsPerThread) {  // a whole half: 16-byte stores
          uint4* dst = reinterpret_cast<uint4*>(logits + static_cast<size_t>(row) * a.vocab + v0);
#pragma unroll
          for (int e = 0; e < kColsPerThread / 8; ++e) {
            uint4 u;
            u.x = pack_bf16x2(acc[8 * e], acc[8 * e + 1]);
            u.y = pack_bf16x2(acc[8 * e + 2], acc[8 * e + 3]);
            u.z = pack_bf16x2(acc[8 * e + 4], acc[8 * e + 5]);
            u.w = pack_bf16x2(acc[8 * e + 6], acc[8 * e + 7]);
            dst[e] = u;
          }
        } else if (logits != nullptr) {  // the vocabulary's last, partial half
          __nv_bfloat16* dst = logits + static_cast<size_t>(row) * a.vocab + v0;
#pragma unroll
          for (int c = 0; c < kColsPerThread; ++c)
            if (c < nv) dst[c] = __float2bfloat16_rn(acc[c]);
        }
        // (max, first argmax, sum of exp(logit - max)) over the existing entries
        float mx = acc[0];
        int am = 0;
#pragma unroll
        for (int c = 1; c < kColsPerThread; ++c)
          if (c < nv && acc[c] > mx) {
            mx = acc[c];
            am = c;
          }
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kColsPerThread; ++c)
          if (c < nv) s4[c & 3] += expf(acc[c] - mx);
        const size_t pi = static_cast<size_t>(2 * vt + half) * a.n_rows + row;
        a.pmax[pi] = mx;
        a.psum[pi] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        a.parg[pi] = v0 + am;
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

// ------------------------------------------------------------ combine
// One warp per row: lane l merges the partials l, l + 32, ... in order, then the 32 lane
// states are merged in lane order (a fixed tree: the result does not depend on timing).  The
// argmax is the lowest vocabulary index among equal maxima.
__global__ void __launch_bounds__(256) lm_combine_kernel(const LmArgs a, int P) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  if (row >= a.n_rows) return;
  float m = -INFINITY, s = 0.f;
  int arg = 0x7fffffff;
  for (int p = lane; p < P; p += 32) {
    const size_t pi = static_cast<size_t>(p) * a.n_rows + row;
    const float mp = a.pmax[pi], sp = a.psum[pi];
    const int ap = a.parg[pi];
    if (mp == -INFINITY) continue;  // an empty partial
    if (mp > m) {
      s = s * expf(m - mp) + sp;  // m = -inf at first: 0 * 0 + sp
      m = mp;
      arg = ap;
    } else {
      s += sp * expf(mp - m);
      if (mp == m && ap < arg) arg = ap;
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {  // merge with the lane o above (lane order)
    const float mo = __shfl_down_sync(0xffffffffu, m, o), so = __shfl_down_sync(0xffffffffu, s, o);
    const int ao = __shfl_down_sync(0xffffffffu, arg, o);
    if (lane + o < 32 && (lane & (2 * o - 1)) == 0) {
      if (mo > m) {
        s = s * expf(m - mo) + so;
        m = mo;
        arg = ao;
      } else if (mo != -INFINITY) {
        s += so * expf(mo - m);
        if (mo == m && ao < arg) arg = ao;
      }
    }
  }
  if (lane == 0) {
    const float L = m + logf(s);
    a.lse[row] = L;
    a.argmax[row] = arg;
    a.p_max[row] = expf(m - L);
  }
}

}  // namespace

// The vocabulary band of the LM head: about 48 MB of W_lm (a third of L2), at least one tile.
int lm_band(int n_vt, int d_model) {
  const long long tile_bytes = static_cast<long long>(kTN) * d_model * 2;
  long long band = (48LL << 20) / tile_bytes;
  band = band < 1 ? 1 : (band > n_vt ? n_vt : band);
  return static_cast<int>(band);
}

size_t lm_head_workspace_bytes(int n_rows, int d_model, int vocab) {
  const size_t P = 2 * static_cast<size_t>((vocab + kTN - 1) / kTN);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return al(static_cast<size_t>(n_rows) * d_model * 2) + 3 * al(P * n_rows * 4);
}

void lm_bind_workspace(LmArgs* a, void* ws) {
  const size_t P = 2 * static_cast<size_t>((a->vocab + kTN - 1) / kTN);
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  uint8_t* p = static_cast<uint8_t*>(ws);
  a->xhat = p;
  p += al(static_cast<size_t>(a->n_rows) * a->d_model * 2);
  a->pmax = reinterpret_cast<float*>(p);
  p += al(P * a->n_rows * 4);
  a->psum = reinterpret_cast<float*>(p);
  p += al(P * a->n_rows * 4);
  a->parg = reinterpret_cast<int32_t*>(p);
}

cudaError_t launch_lm_head(const void* w_lm, const LmArgs& a, int num_sms, cudaStream_t stream) {
  if (a.n_rows <= 0) return cudaSuccess;
  const int n_vt = (a.vocab + kTN - 1) / kTN, n_tt = (a.n_rows + kTM - 1) / kTM;
  const int P = 2 * n_vt;
  CUtensorMap tm_w, tm_x;
  cudaError_t e = encode_2d_sw128(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_lm, a.d_model, a.vocab, kBK, kTN);
  if (e == cudaSuccess)
    e = encode_2d_sw128(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.xhat, a.d_model, a.n_rows, kBK, kTM);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, lm_head_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;  // the register split assumes it
  e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  if (e != cudaSuccess) return e;
  auto launch = [&](auto kern, dim3 grid, int threads, int smem, auto... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
  };
  const int warps_blocks = (a.n_rows * 32 + 255) / 256;
  e = launch(lm_gather_norm_kernel, dim3(warps_blocks), 256, 0, a);
  if (e != cudaSuccess) return e;
  const int n_tiles = n_vt * n_tt;
  e = launch(lm_head_kernel, dim3(n_tiles < num_sms ? n_tiles : num_sms), kThreads, kDynSmem, tm_w, tm_x, a, n_vt,
             n_tt, lm_band(n_vt, a.d_model));
  if (e != cudaSuccess) return e;
  return launch(lm_combine_kernel, dim3(warps_blocks), 256, 0, a, P);
}

}  // namespace dllm
