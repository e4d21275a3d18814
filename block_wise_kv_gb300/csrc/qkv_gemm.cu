// qkv_gemm.cu — fused QKV projection + RoPE + single cache write (sm_103a).
//
// Computes, for a set of token rows t with normalised input x^_t (bf16, the
// output of the RMSNorm kernel), y_t = W_qkv x^_t with fp32 accumulation,
// rotates the q and k parts (RoPE, rotate-half pairs (i, i + d/2) at the
// token's absolute position) and writes q, k, v once, as bf16, to their
// destinations: k, v into the paged pools through the block table, q into
// q_block (inner step) or q_pool (block boundary).  This is the Flash-Cache
// fusion of the Flash-dLLM write-up ("Flash-Cache: Fusing Projection, RoPE,
// and Cache Writes into One Kernel": projection and RoPE on chip, keys and
// values written straight into the cache in one HBM write) applied to the
// token-wise operators of LaCache §3.3.2, Eq. (1).
//
// GB300 design.  The contraction is "swap-AB": the 128-row weight tiles are
// the tcgen05 M operand and the (few) token rows are the N operand, so a
// 32-token inner step still fills a 128 x 32 UMMA.  A warp issues TMA loads of
// 128 x 64 weight tiles and BN x 64 token tiles (128-byte swizzle) into a
// multi-stage mbarrier ring; one thread issues tcgen05.mma into a TMEM
// accumulator.  When the weight-tile x token-tile grid alone cannot fill the
// 152 SMs (the inner step is bound by streaming the 100 MB weight matrix),
// the K dimension is split across the CTAs of a thread-block cluster and the
// fp32 partial tiles are summed through distributed shared memory before the
// RoPE epilogue, so nothing but the final bf16 q/k/v leaves the chip.
#include <cooperative_groups.h>

#include "kernels.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace cg = cooperative_groups;

namespace dllm {
namespace {

constexpr int kThreads = 128;
constexpr int kTileM = 128;     // weight rows per tile (UMMA M)
constexpr int kTileK = 64;      // K elements per stage (one 128-byte swizzle row)
constexpr int kTileABytes = kTileM * kTileK * 2;

template <int BN>
struct GemmCfg;
template <>
struct GemmCfg<32> {
  static constexpr int kStages = 5;
};
template <>
struct GemmCfg<64> {
  static constexpr int kStages = 4;
};
template <>
struct GemmCfg<128> {
  static constexpr int kStages = 4;
};
template <>
struct GemmCfg<256> {
  static constexpr int kStages = 4;
};

template <int BN>
constexpr int gemm_smem_bytes() {
  return GemmCfg<BN>::kStages * (kTileABytes + BN * kTileK * 2) + 1024;
}

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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                    const QkvArgs a) {
  constexpr int kStages = GemmCfg<BN>::kStages;
  constexpr int kTileBBytes = BN * kTileK * 2;
  constexpr int kStageBytes = kTileABytes + kTileBBytes;
  constexpr uint32_t kTmemCols = BN;  // power of two >= 32

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], tmem_full_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ long long tok_kv[BN];   // element offset of (page, head 0, slot) in the pools, -1: no write
  __shared__ long long tok_q[BN];    // element offset of the q destination for head 0, -1: no write
  __shared__ int tok_pos[BN];        // absolute position (RoPE)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = gridDim.x, rank = blockIdx.x;
  const int mt = blockIdx.y, nt = blockIdx.z;
  const int nkb_total = a.d_model / kTileK;
  const int kb0 = rank * nkb_total / S, kb1 = (rank + 1) * nkb_total / S;
  const int nkb = kb1 - kb0;
  const BatchArgs& bt = a.bt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tmem_full_bar, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 2) tmem_alloc(&tmem_base_sh, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (i >= kStages && !mbar_wait(&empty_bar[s], ph ^ 1)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        uint8_t* sa = smem + s * kStageBytes;
        mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        tma_load_2d(sa, &tm_w, &full_bar[s], (kb0 + i) * kTileK, mt * kTileM);
        tma_load_2d(sa + kTileABytes, &tm_x, &full_bar[s], (kb0 + i) * kTileK, nt * BN);
        ++issued;
      }
      // Drain: every issued load has landed before the CTA can retire.
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % kStages], (i / kStages) & 1)) report_error(bt.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = umma_idesc_bf16(kTileM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(&full_bar[s], ph)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * kStageBytes), sb = sa + kTileABytes;
#pragma unroll
        for (int k = 0; k < kTileK / 16; ++k)
          umma_bf16(tmem, umma_desc_sw128(sa + k * 32), umma_desc_sw128(sb + k * 32), idesc, (i | k) != 0);
        umma_commit(&empty_bar[s]);
      }
      umma_commit(&tmem_full_bar);
    }
  } else {
    // ---- warps 2-3: resolve each token column to its destinations while the
    // main loop runs.
    const int H = a.n_heads, d = a.head_dim;
    for (int c = threadIdx.x - 64; c < BN; c += 64) {
      long long kv = -1, qd = -1;
      int pos = 0;
      const int j = nt * BN + c;
      if (j < a.n_tok) {
        const int32_t* cu = a.mode == kModeBlock ? bt.cu_block : bt.cu_seq;
        const int b = find_seq(cu, bt.batch, j);
        const int off = j - __ldg(cu + b);
        const int nb = __ldg(bt.seq_len + b), sb = __ldg(bt.block_start + b), lb = __ldg(bt.block_len + b);
        pos = a.mode == kModeBlock ? sb + off : off;
        const bool shape_ok = nb >= 1 && nb <= bt.max_seq_len && lb >= 1 && lb <= bt.max_block_len && sb >= 0 &&
                              sb + lb <= nb && (a.mode == kModeBlock ? off < lb : off < nb) && pos >= 0 &&
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
            else if (pos < sb || pos >= sb + lb)
              qd = kv;  // queries are cached for the invariant rows only
          }
        }
      }
      tok_kv[c] = kv;
      tok_q[c] = qd;
      tok_pos[c] = pos;
    }
  }
  __syncwarp();

  // ---- accumulator: TMEM -> shared (token-major partial tile [BN][128])
  if (!mbar_wait(&tmem_full_bar, 0)) report_error(bt.err, kErrTimeout);
  tc_fence_after();
  float* part = reinterpret_cast<float*>(smem);  // reuses the drained pipeline buffers
  {
    const int row = warp * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, v);
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) part[(c0 + jj) * kTileM + row] = v[jj];
    }
  }
  tc_fence_before();
  cg::cluster_group cluster = cg::this_cluster();
  if (S > 1)
    cluster.sync();
  else
    __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);

  // ---- epilogue: sum the split-K partials of this rank's token columns,
  // rotate q/k, round to bf16 and write each value once.
  {
    const int H = a.n_heads, d = a.head_dim, half = d >> 1;
    const int HD = H * d;
    const int grow0 = mt * kTileM;
    const int which = grow0 / HD;                // 0: q, 1: k, 2: v
    const int head0 = (grow0 % HD) / d;
    const int ncols = min(BN, a.n_tok - nt * BN);
    const int nmine = ncols > rank ? (ncols - rank + S - 1) / S : 0;
    __nv_bfloat16* kpool = static_cast<__nv_bfloat16*>(a.k_pool);
    __nv_bfloat16* vpool = static_cast<__nv_bfloat16*>(a.v_pool);
    __nv_bfloat16* qdst = static_cast<__nv_bfloat16*>(a.mode == kModeBlock ? a.q_block : a.q_pool);
    for (int item = threadIdx.x; item < nmine * 64; item += kThreads) {
      const int c = rank + S * (item >> 6);
      const int jp = item & 63;
      const long long kv = tok_kv[c];
      if (kv < 0) continue;
      const int hit = jp / half, t = jp % half;
      const int row_lo = hit * d + t, row_hi = row_lo + half;
      float lo = 0.f, hi = 0.f;
      for (int r = 0; r < S; ++r) {
        const float* p = S > 1 ? cluster.map_shared_rank(part, r) : part;
        lo += p[c * kTileM + row_lo];
        hi += p[c * kTileM + row_hi];
      }
      const int head = head0 + hit;
      __nv_bfloat16* out;
      if (which == 2) {
        out = vpool + kv + static_cast<long long>(head) * kPage * d;
      } else {
        const float2 cs = *reinterpret_cast<const float2*>(a.rope + (static_cast<size_t>(tok_pos[c]) * half + t) * 2);
        const float rlo = lo * cs.x - hi * cs.y;
        const float rhi = hi * cs.x + lo * cs.y;
        lo = rlo;
        hi = rhi;
        if (which == 1) {
          out = kpool + kv + static_cast<long long>(head) * kPage * d;
        } else {
          const long long qd = tok_q[c];
          if (qd < 0) continue;
          out = qdst + qd + static_cast<long long>(head) * (a.mode == kModeBlock ? d : kPage * d);
        }
      }
      out[t] = __float2bfloat16_rn(lo);
      out[t + half] = __float2bfloat16_rn(hi);
    }
  }
  if (S > 1) cluster.sync();  // peers may still read this CTA's partial tile
}

template <int BN>
cudaError_t launch_bn(const void* w_qkv, const void* xhat, const QkvArgs& a, int num_sms, cudaStream_t stream) {
  const int HD = a.n_heads * a.head_dim;
  CUtensorMap tm_w, tm_x;
  cudaError_t e = encode_2d_sw128(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_qkv, a.d_model, 3ull * HD, kTileK,
                                  kTileM);
  if (e != cudaSuccess) return e;
  e = encode_2d_sw128(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xhat, a.d_model, a.n_tok, kTileK, BN);
  if (e != cudaSuccess) return e;

  const int n_wt = 3 * HD / kTileM;
  const int n_tt = (a.n_tok + BN - 1) / BN;
  const int nkb = a.d_model / kTileK;
  const int smem = gemm_smem_bytes<BN>();
  const int per_sm = (228 * 1024) / (smem + 2048);
  const long long tiles = static_cast<long long>(n_wt) * n_tt;
  const long long slots = static_cast<long long>(num_sms) * (per_sm > 0 ? per_sm : 1);
  int split = 1;
  if (tiles < slots) {
    split = static_cast<int>(slots / tiles);
    if (split > 8) split = 8;
    if (split > nkb / 2) split = nkb / 2;
    if (split < 1) split = 1;
  }

  auto kern = qkv_gemm_kernel<BN>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split, n_wt, n_tt);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, a);
}

}  // namespace

cudaError_t launch_qkv_gemm(const void* w_qkv, const void* xhat, const QkvArgs& a, int num_sms,
                            cudaStream_t stream) {
  if (a.n_tok <= 0) return cudaSuccess;
  if (a.n_tok <= 32) return launch_bn<32>(w_qkv, xhat, a, num_sms, stream);
  if (a.n_tok <= 64) return launch_bn<64>(w_qkv, xhat, a, num_sms, stream);
  if (a.n_tok <= 128) return launch_bn<128>(w_qkv, xhat, a, num_sms, stream);
  return launch_bn<256>(w_qkv, xhat, a, num_sms, stream);
}

}  // namespace dllm
