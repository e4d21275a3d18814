// ffn.cu — the rest of the layer for the current blocks' rows (sm_103a): the
// attention output projection with its residual, then the FFN with per-group
// FP8 ("LaCache: Exact Caching and Precision-Adaptive Inference for Diffusion
// Large Language Models", §3.4 Mixed precision strategy, Eq. (7)-(8): a
// tensor split into groups is quantised as x' = clip(x / scale_g) with
// scale_g = max_g |x| / Q_max; the quantisation is fused into the AddNorm
// before the gate-up linear and into the SwiGLU before the down linear).
//
//   h1 = x + O W_o^T                     (bf16 GEMM; O the block rows of the attention output)
//   x2 = RMSNorm(h1) g2 -> e4m3 codes, one scale per (row, 128 columns)      (AddNorm + quant)
//   a  = SiLU(x2 W_gate^T) * (x2 W_up^T) -> e4m3, one scale per (row, 128)  (FP8 GEMM + SwiGLU)
//   y  = h1 + a W_down^T                                                     (FP8 GEMM + residual)
//
// The weights of the FP8 GEMMs are e4m3 with one fp32 scale per 128 x 128
// block.  Every GEMM is one token-major tcgen05 kernel: tiles of 128 rows
// (M) x 256 weight rows (N), K in chunks of 128 (one quantisation group):
// the tensor core sums a chunk into TMEM (kind::f16 for bf16,
// kind::f8f6f4 for e4m3) and warps 4-11 add it into fp32 registers times the
// chunk's two scales (row group x weight block), so the dequantisation is
// exact per group.  A thread holds one row and 128 weight rows.  Few tiles
// (the projections to d_model at a few hundred rows) split K over the CTAs:
// fp32 partials per split, summed in split order with the residual by a
// reduction kernel.
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
constexpr int kTN = 256;                 // weight rows per tile (tcgen05 N)
constexpr int kRowBytes = 128;           // bytes of K per ring stage and row (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kABytes = kTM * kRowBytes;  // 16 KB
constexpr int kBBytes = kTN * kRowBytes;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kDynSmem = kStages * kStageBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr int kColsPerThread = kTN / 2;
constexpr int kAcc = kAccWarps * 32;
constexpr float kE4m3Max = 448.f;        // Q_max of e4m3

constexpr int kEpiPartial = 0;  // fp32 partial sums of a K split
constexpr int kEpiSwiGLU = 1;   // SiLU(gate) * up of interleaved rows, quantised to e4m3 per 128 units

// ------------------------------------------------------------ gather
// Block row j of the attention output: row cu_seq[b] + s_b + i of o_full.
// The sequence of block row j: the largest b with cu_block[b] <= j, found by the warp 32
// sequences at a time (cu_block is increasing; every lane gets the same answer).
__device__ __forceinline__ int warp_find_seq(const int32_t* cu, int batch, int j, int lane) {
  int count = 0;
  for (int b0 = 0; b0 < batch; b0 += 32) {
    const int b = b0 + lane;
    const unsigned le = __ballot_sync(0xffffffffu, b < batch && __ldg(cu + b) <= j);
    count += __popc(le);
    if (le != 0xffffffffu) break;
  }
  return count > 0 ? count - 1 : 0;
}

constexpr int kRowThreads = 128;  // the row kernels: four warps, one row each

__global__ void __launch_bounds__(kRowThreads) ffn_gather_kernel(const FfnArgs a) {
  const int j = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  const BatchArgs& bt = a.bt;
  if (j >= a.n_rows) return;
  const int b = warp_find_seq(bt.cu_block, bt.batch, j, lane), off = j - __ldg(bt.cu_block + b);
  const int nb = __ldg(bt.seq_len + b), sb = __ldg(bt.block_start + b), lb = __ldg(bt.block_len + b);
  const int cus = __ldg(bt.cu_seq + b);
  const int nvec = a.hd / 8;
  uint4* dst = static_cast<uint4*>(a.o_block) + static_cast<size_t>(j) * nvec;
  const bool ok = nb >= 1 && nb <= bt.max_seq_len && lb >= 1 && lb <= bt.max_block_len && sb >= 0 && sb + lb <= nb &&
                  off >= 0 && off < lb && cus >= 0 && cus + nb <= bt.total_seq_rows;
  if (!ok) {
    if (lane == 0) report_error(bt.err, kErrBadShape);
    for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* src = static_cast<const uint4*>(a.o_full) + static_cast<size_t>(cus + sb + off) * nvec;
  for (int v0 = 0; v0 < nvec; v0 += 32 * 8) {  // eight 16-byte loads in flight a lane, then the stores
    uint4 t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = v0 + lane + 32 * i;
      if (v < nvec) t[i] = __ldg(src + v);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int v = v0 + lane + 32 * i;
      if (v < nvec) dst[v] = t[i];
    }
  }
}

// ------------------------------------------------------------ AddNorm + quantisation
// One warp per row of h1: x2 = RMSNorm(h1) g2 in fp32 (the exact sum of squares and scale of
// the projection's RMSNorm), then per group of 128 columns scale = max |x2| / 448 and the e4m3
// codes of x2 / scale (round to nearest even).  A lane holds the 16-byte pieces lane + 32 i of
// the row, so a group of 128 columns is the 16 pieces of one half-warp in one round.
constexpr int kRowPieces = 16;  // pieces a lane keeps in registers (rows up to 4096 wide)

// Eight values of x2 (piece hu of h1, gain piece gu), their group's scale over the half-warp,
// and their eight e4m3 codes; the lane at the start of the half writes the scale.
__device__ __forceinline__ uint2 quant_piece(const uint4& hu, const uint4& gu, float inv, float* scale_out,
                                             bool writes_scale) {
  const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&hu);
  const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gu);
  float v[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 h = __bfloat1622float2(hp[i]), g = __bfloat1622float2(gp[i]);
    v[2 * i] = h.x * inv * g.x;
    v[2 * i + 1] = h.y * inv * g.y;
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = amax / kE4m3Max;  // Eq. (8)
  if (writes_scale) *scale_out = sc;
  uint32_t w[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {  // Eq. (7)
    const int c = 4 * k;
    const uint16_t p0 = sc > 0.f ? cvt_e4m3x2(__fdiv_rn(v[c], sc), __fdiv_rn(v[c + 1], sc)) : 0;
    const uint16_t p1 = sc > 0.f ? cvt_e4m3x2(__fdiv_rn(v[c + 2], sc), __fdiv_rn(v[c + 3], sc)) : 0;
    w[k] = static_cast<uint32_t>(p0) | (static_cast<uint32_t>(p1) << 16);
  }
  return make_uint2(w[0], w[1]);
}

__global__ void __launch_bounds__(kRowThreads) ffn_addnorm_quant_kernel(const FfnArgs a) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  if (row >= a.n_rows) return;
  const int D = a.d_model, nvec = D / 8, ng = D / 128;
  const uint4* hr = static_cast<const uint4*>(a.h1) + static_cast<size_t>(row) * nvec;
  const uint4* gr = static_cast<const uint4*>(a.gain2);
  uint2* q = reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.x2) + static_cast<size_t>(row) * D);
  float* scales = a.x2_scale + static_cast<size_t>(row) * ng;
  const bool held = nvec <= 32 * kRowPieces;
  uint4 hv[kRowPieces];
  float shi = 0.f, slo = 0.f;  // exact sum of squares as a float pair, pieces in order
  if (held) {
#pragma unroll
    for (int i = 0; i < kRowPieces; ++i)
      if (lane + 32 * i < nvec) hv[i] = hr[lane + 32 * i];
#pragma unroll
    for (int i = 0; i < kRowPieces; ++i)
      if (lane + 32 * i < nvec) sumsq_pair_add(hv[i], shi, slo);
  } else {
    for (int v = lane; v < nvec; v += 32) sumsq_pair_add(hr[v], shi, slo);
  }
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, shi, o), ol = __shfl_xor_sync(0xffffffffu, slo, o);
    pair_add(shi, slo, oh, ol);
  }
  float y_hi = 0.f, y_lo = 0.f;
  if (lane == 0) {
    two_sum(shi, slo, shi, slo);
    rsqrt_pair(shi, slo, D, a.rms_eps, y_hi, y_lo);
  }
  const float inv = __shfl_sync(0xffffffffu, y_hi, 0) + __shfl_sync(0xffffffffu, y_lo, 0);
  // nvec is a multiple of 16, so a half-warp's 16 pieces are all in the row or all past it
  const bool first_of_group = (lane & 15) == 0;
  if (held) {
#pragma unroll
    for (int i = 0; i < kRowPieces; ++i) {
      if (32 * i >= nvec) break;
      const int v = lane + 32 * i;
      const bool on = v < nvec;
      const uint2 c = quant_piece(on ? hv[i] : make_uint4(0u, 0u, 0u, 0u), on ? __ldg(gr + v) : make_uint4(0u, 0u, 0u, 0u),
                                  inv, scales + (v >> 4), on && first_of_group);
      if (on) q[v] = c;
    }
  } else {
    for (int v0 = 0; v0 < nvec; v0 += 32) {
      const int v = v0 + lane;
      const bool on = v < nvec;
      const uint2 c = quant_piece(on ? hr[v] : make_uint4(0u, 0u, 0u, 0u), on ? __ldg(gr + v) : make_uint4(0u, 0u, 0u, 0u),
                                  inv, scales + (v >> 4), on && first_of_group);
      if (on) q[v] = c;
    }
  }
}

// Tile order: weight tiles in bands of `band` (the last may be narrower); within a band, row
// tile by row tile, weight tile fastest.
__device__ __forceinline__ void dense_tile_coords(int tile, int n_nt, int n_mt, int band, int& nt, int& mt) {
  const int full = n_nt / band;
  const int in_full = full * band * n_mt;
  if (tile < in_full) {
    const int bi = tile / (band * n_mt), r = tile % (band * n_mt);
    mt = r / band;
    nt = bi * band + r % band;
  } else {
    const int rest = n_nt - full * band, r = tile - in_full;
    mt = r / rest;
    nt = full * band + r % rest;
  }
}

// ------------------------------------------------------------ the GEMMs
template <bool FP8, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    dense_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const DenseArgs g, int n_nt, int n_mt, int band) {
  constexpr uint32_t kIdesc = FP8 ? umma_idesc_e4m3(kTM, kTN) : umma_idesc_bf16(kTM, kTN);
  constexpr int kStagesPerChunk = FP8 ? 1 : 2;  // a chunk of K = 128 elements
  constexpr int kStageK = FP8 ? 128 : 64;       // elements of K per stage (128 bytes a row)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float amax_sh[2][kTM];  // SwiGLU: each half's group max of a row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nck = g.K / 128, S = g.splits;
  const int G = static_cast<int>(gridDim.x);
  const int n_units = n_nt * n_mt * S;

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
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  griddep_launch_dependents();
  // unit u: tile u / S (in band order), K split u % S: chunks [s nck / S, (s + 1) nck / S)
  auto unit = [&](int u, int& nt, int& mt, int& c0, int& c1) {
    dense_tile_coords(u / S, n_nt, n_mt, band, nt, mt);
    const int s = u % S;
    c0 = s * nck / S;
    c1 = (s + 1) * nck / S;
  };

  if (warp < kFirstAccWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFewRegs));
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        griddep_wait();  // the rows come from the preceding kernel
        int q = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += G) {
          int nt, mt, c0, c1;
          unit(u, nt, mt, c0, c1);
          for (int kb = c0 * kStagesPerChunk; kb < c1 * kStagesPerChunk; ++kb, ++q) {
            const int s = q % kStages;
            if (q >= kStages && !mbar_wait(&empty_bar[s], ((q / kStages) - 1) & 1)) {
              report_error(g.err, kErrTimeout);
              ok = false;
              break;
            }
            uint8_t* st = smem + s * kStageBytes;
            mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
            tma_load_2d(st, &tm_a, &full_bar[s], kb * kStageK, mt * kTM);            // rows past M read 0
            tma_load_2d(st + kABytes, &tm_b, &full_bar[s], kb * kStageK, nt * kTN);  // rows past N read 0
          }
        }
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report_error(g.err, kErrTimeout);
        for (int i = (q > kStages ? q - kStages : 0); i < q; ++i)
          if (!mbar_wait(&empty_bar[i % kStages], (i / kStages) & 1)) report_error(g.err, kErrTimeout);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        int q = 0, nc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += G) {
          int nt, mt, c0, c1;
          unit(u, nt, mt, c0, c1);
          for (int ck = c0; ck < c1 && ok; ++ck, ++nc) {
            const int b = nc & 1;
            if (nc >= 2 && !mbar_wait(&tempty_bar[b], ((nc >> 1) - 1) & 1)) {
              report_error(g.err, kErrTimeout);
              ok = false;
              break;
            }
            const uint32_t d = tmem + static_cast<uint32_t>(b * kTN);
            for (int hb = 0; hb < kStagesPerChunk; ++hb, ++q) {
              const int s = q % kStages;
              if (!mbar_wait(&full_bar[s], (q / kStages) & 1)) {
                report_error(g.err, kErrTimeout);
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sa = smem_u32(smem + s * kStageBytes), sb = sa + kABytes;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of K per instruction
                if (FP8)
                  umma_e4m3(d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), kIdesc,
                            (hb > 0 || kk > 0) ? 1u : 0u);
                else
                  umma_bf16(d, umma_desc_sw128(sa + kk * 32), umma_desc_sw128(sb + kk * 32), kIdesc,
                            (hb > 0 || kk > 0) ? 1u : 0u);
              }
              umma_commit(&empty_bar[s]);
            }
            if (!ok) break;
            umma_commit(&tfull_bar[b]);
          }
        }
        if (!ok)
          for (int b = 0; b < 2; ++b) umma_commit(&tfull_bar[b]);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kManyRegs));
    // ------------------------------------------------------------ accumulator warps
    // The rows' group scales come from the preceding kernel (the AddNorm, the SwiGLU
    // epilogue): read only once it has completed.
    griddep_wait();
    const int ai = warp - kFirstAccWarp;
    const int quad = warp & 3;
    const int half = ai >> 2;  // the 128 weight rows of a tile this thread holds
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int nkg = g.K / 128;
    float acc[kColsPerThread];
#pragma unroll
    for (int c = 0; c < kColsPerThread; ++c) acc[c] = 0.f;
    bool ok = true;
    int nc = 0;
    for (int u = blockIdx.x; u < n_units; u += G) {
      int nt, mt, c0, c1;
      unit(u, nt, mt, c0, c1);
      const int rt = quad * 32 + lane;  // row of the tile
      const int row = mt * kTM + rt;
      const int nblk = nt * 2 + half;   // the weight block (128 rows) of this thread
      const bool row_ok = row < g.M, blk_ok = nblk * 128 < g.N;
      // The chunk's dequantisation f = row group scale x weight block scale; the pair is
      // loaded a chunk ahead of its use (its latency would otherwise stall every chunk).
      auto ld_sa = [&](int ck) { return row_ok && ck < c1 ? g.sa[static_cast<size_t>(row) * nkg + ck] : 0.f; };
      auto ld_sb = [&](int ck) { return blk_ok && ck < c1 ? g.sb[static_cast<size_t>(nblk) * nkg + ck] : 0.f; };
      float sa0 = 1.f, sb0 = 1.f;
      if (FP8) sa0 = ld_sa(c0), sb0 = ld_sb(c0);
      for (int ck = c0; ck < c1; ++ck, ++nc) {
        float sa1 = 1.f, sb1 = 1.f;
        if (FP8) sa1 = ld_sa(ck + 1), sb1 = ld_sb(ck + 1);
        const float f = FP8 ? sa0 * sb0 : 1.f;
        const int b = nc & 1;
        if (ok && !mbar_wait(&tfull_bar[b], (nc >> 1) & 1)) {
          report_error(g.err, kErrTimeout);
          ok = false;
        }
        tc_fence_after();
#pragma unroll
        for (int cq = 0; cq < kColsPerThread; cq += 64) {  // two TMEM loads in flight per wait
          float v[64];
          tmem_ld_32x32b_x64(lane_base + static_cast<uint32_t>(b * kTN + half * kColsPerThread + cq), v);
#pragma unroll
          for (int i = 0; i < 64; ++i) acc[cq + i] = fmaf(v[i], f, acc[cq + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
        sa0 = sa1, sb0 = sb1;
      }
      const int n0 = nblk * 128;
      if (EPI == kEpiPartial) {
        // fp32 partial of split u % S for this row and 128 weight rows
        if (row_ok && blk_ok) {
          float4* dst =
              reinterpret_cast<float4*>(g.part + (static_cast<size_t>(u % S) * g.M + row) * g.N + n0);
#pragma unroll
          for (int e = 0; e < kColsPerThread / 4; ++e)
            dst[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
        }
      } else {
        // SwiGLU: weight rows 2j (gate) and 2j + 1 (up) of hidden unit j; this thread holds
        // units n0 / 2 .. n0 / 2 + 63, the tile's 128 units (one quantisation group) are
        // shared with the other half's thread of the same row
        float av[kColsPerThread / 2];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < kColsPerThread / 2; ++j) {
          const float gt = acc[2 * j], up = acc[2 * j + 1];
          av[j] = gt / (1.f + expf(-gt)) * up;
          amax = fmaxf(amax, fabsf(av[j]));
        }
        amax_sh[half][rt] = amax;
        named_barrier(1, kAcc);
        amax = fmaxf(amax_sh[0][rt], amax_sh[1][rt]);
        named_barrier(1, kAcc);  // read before the next tile writes
        const float sc = amax / kE4m3Max;  // Eq. (8)
        const int F = g.N / 2, ngf = F / 128;
        if (row_ok && blk_ok) {
          if (half == 0) g.out_scale[static_cast<size_t>(row) * ngf + nt] = sc;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(g.out8) + static_cast<size_t>(row) * F +
                                                 nt * 128 + half * 64);
#pragma unroll
          for (int e = 0; e < 4; ++e) {  // Eq. (7): 16 codes per 16-byte store
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = 16 * e + 4 * k;
              const uint16_t p0 = sc > 0.f ? cvt_e4m3x2(__fdiv_rn(av[c], sc), __fdiv_rn(av[c + 1], sc)) : 0;
              const uint16_t p1 = sc > 0.f ? cvt_e4m3x2(__fdiv_rn(av[c + 2], sc), __fdiv_rn(av[c + 3], sc)) : 0;
              w[k] = static_cast<uint32_t>(p0) | (static_cast<uint32_t>(p1) << 16);
            }
            dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
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

// out[r][n] = bf16(sum over splits s of part[s][r][n] + residual[r][n]), splits in order.
__global__ void __launch_bounds__(256) dense_reduce_kernel(const DenseArgs g, const void* residual, void* out) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t i4 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // 4 elements each
  const size_t n = static_cast<size_t>(g.M) * g.N;
  if (i4 * 4 >= n) return;
  const float4* p = reinterpret_cast<const float4*>(g.part);
  float4 s = p[i4];
  for (int k = 1; k < g.splits; ++k) {
    const float4 t = p[k * (n / 4) + i4];
    s.x += t.x;
    s.y += t.y;
    s.z += t.z;
    s.w += t.w;
  }
  const uint2 rr = reinterpret_cast<const uint2*>(residual)[i4];
  const __nv_bfloat162 r0 = *reinterpret_cast<const __nv_bfloat162*>(&rr.x);
  const __nv_bfloat162 r1 = *reinterpret_cast<const __nv_bfloat162*>(&rr.y);
  uint2 o;
  o.x = pack_bf16x2(s.x + __low2float(r0), s.y + __high2float(r0));
  o.y = pack_bf16x2(s.z + __low2float(r1), s.w + __high2float(r1));
  reinterpret_cast<uint2*>(out)[i4] = o;
}

}  // namespace

namespace {
// K splits of a GEMM with n_tiles output tiles: enough units for every SM, at most one per chunk.
int dense_splits(int n_tiles, int nck, int num_sms) {
  int s = (num_sms + n_tiles - 1) / n_tiles;
  return s < 1 ? 1 : (s > nck ? nck : s);
}
size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
struct FfnPlan {
  int s_o, s_d;  // K splits of the output projection and of the down GEMM
  size_t o_block, h1, x2, x2s, a8, as, part, total;  // workspace offsets
};
FfnPlan ffn_plan(int M, int D, int HD, int F, int num_sms) {
  FfnPlan p;
  const int mt = (M + kTM - 1) / kTM, nt_d = (D + kTN - 1) / kTN;
  p.s_o = dense_splits(mt * nt_d, HD / 128, num_sms);
  p.s_d = dense_splits(mt * nt_d, F / 128, num_sms);
  const int s = p.s_o > p.s_d ? p.s_o : p.s_d;
  size_t at = 0;
  p.o_block = at;
  at += al256(static_cast<size_t>(M) * HD * 2);
  p.h1 = at;
  at += al256(static_cast<size_t>(M) * D * 2);
  p.x2 = at;
  at += al256(static_cast<size_t>(M) * D);
  p.x2s = at;
  at += al256(static_cast<size_t>(M) * (D / 128) * 4);
  p.a8 = at;
  at += al256(static_cast<size_t>(M) * F);
  p.as = at;
  at += al256(static_cast<size_t>(M) * (F / 128) * 4);
  p.part = at;
  at += al256(static_cast<size_t>(s) * M * D * 4);
  p.total = at;
  return p;
}

template <class K, class... Args>
cudaError_t launch_ex(K kern, int grid, int threads, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// One GEMM: A [M][K] (bf16, or e4m3 codes), B [N][K] likewise, in tiles of 128 x 256.
template <bool FP8, int EPI>
cudaError_t launch_dense(const void* A, const void* B, DenseArgs g, int num_sms, cudaStream_t stream) {
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int eb = FP8 ? 1 : 2, box = kRowBytes / eb;
  CUtensorMap tm_a, tm_b;
  cudaError_t e = encode_2d_sw128(&tm_a, dt, eb, A, g.K, g.M, box, kTM);
  if (e == cudaSuccess) e = encode_2d_sw128(&tm_b, dt, eb, B, g.K, g.N, box, kTN);
  if (e != cudaSuccess) return e;
  auto kern = dense_kernel<FP8, EPI>;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;  // the register split assumes it
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  if (e != cudaSuccess) return e;
  const int n_nt = (g.N + kTN - 1) / kTN, n_mt = (g.M + kTM - 1) / kTM;
  const int units = n_nt * n_mt * g.splits;
  const long long tile_bytes = static_cast<long long>(kTN) * g.K * eb;
  long long band = (48LL << 20) / tile_bytes;  // weight tiles of about 48 MB stay in L2
  band = band < 1 ? 1 : (band > n_nt ? n_nt : band);
  return launch_ex(kern, units < num_sms ? units : num_sms, kThreads, kDynSmem, stream, tm_a, tm_b, g, n_nt, n_mt,
                   static_cast<int>(band));
}

cudaError_t launch_reduce(const DenseArgs& g, const void* residual, void* out, cudaStream_t stream) {
  const size_t n4 = static_cast<size_t>(g.M) * g.N / 4;
  return launch_ex(dense_reduce_kernel, static_cast<int>((n4 + 255) / 256), 256, 0, stream, g, residual, out);
}
}  // namespace

size_t ffn_workspace_bytes(int n_rows, int d_model, int hd, int d_ff, int num_sms) {
  return ffn_plan(n_rows, d_model, hd, d_ff, num_sms).total;
}

cudaError_t launch_ffn(const FfnArgs& a0, const FfnWeights& w, void* ws, int num_sms, cudaStream_t stream) {
  if (a0.n_rows <= 0) return cudaSuccess;
  const int M = a0.n_rows, D = a0.d_model, HD = a0.hd, F = a0.d_ff;
  const FfnPlan p = ffn_plan(M, D, HD, F, num_sms);
  uint8_t* base = static_cast<uint8_t*>(ws);
  FfnArgs a = a0;
  a.o_block = base + p.o_block;
  a.h1 = base + p.h1;
  a.x2 = base + p.x2;
  a.x2_scale = reinterpret_cast<float*>(base + p.x2s);
  float* part = reinterpret_cast<float*>(base + p.part);
  uint8_t* a8 = base + p.a8;
  float* as = reinterpret_cast<float*>(base + p.as);
  const int warp_blocks = (M * 32 + kRowThreads - 1) / kRowThreads;  // a warp per row
  // the block rows of the attention output
  cudaError_t e = launch_ex(ffn_gather_kernel, warp_blocks, kRowThreads, 0, stream, a);
  if (e != cudaSuccess) return e;
  // h1 = x + O W_o^T
  DenseArgs g = {M, D, HD, p.s_o, nullptr, nullptr, part, nullptr, nullptr, a.bt.err};
  e = launch_dense<false, kEpiPartial>(a.o_block, w.w_o, g, num_sms, stream);
  if (e == cudaSuccess) e = launch_reduce(g, a.x_block, a.h1, stream);
  if (e != cudaSuccess) return e;
  // x2 = quant(RMSNorm(h1) g2)
  e = launch_ex(ffn_addnorm_quant_kernel, warp_blocks, kRowThreads, 0, stream, a);
  if (e != cudaSuccess) return e;
  // a = quant(SiLU(gate) * up)
  DenseArgs gu = {M, 2 * F, D, 1, a.x2_scale, w.gu_scale, nullptr, a8, as, a.bt.err};
  e = launch_dense<true, kEpiSwiGLU>(a.x2, w.w_gu, gu, num_sms, stream);
  if (e != cudaSuccess) return e;
  // y = h1 + a W_down^T
  DenseArgs dn = {M, D, F, p.s_d, as, w.down_scale, part, nullptr, nullptr, a.bt.err};
  e = launch_dense<true, kEpiPartial>(a8, w.w_down, dn, num_sms, stream);
  if (e == cudaSuccess) e = launch_reduce(dn, a.h1, a.y, stream);
  return e;
}

}  // namespace dllm
