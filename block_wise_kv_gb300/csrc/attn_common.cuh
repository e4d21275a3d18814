// attn_common.cuh — device building blocks shared by the attention kernels
// (sm_103a): 128-byte-swizzled tile addressing, the warp-level online-softmax
// step on mma.sync m16n8k16 (bf16 in, fp32 accumulate), per-sequence metadata
// checks, and the launch helpers.
//
// The online softmax works in base 2: scores are pre-multiplied by
// scale * log2(e) and every m kept on chip is in those units; the ABI's
// m_pool and lse are natural-log units.
#pragma once

#include "kernels.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace dllm {
namespace attn {

constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x on the SFU (ex2.approx: relative error ~2^-22, ftz), used for softmax weights.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of (row, 16-byte chunk) in a 64-row bf16 tile of D columns,
// stored as D/64 column halves of 64 x 128 B written by TMA with 128-byte
// swizzling (each half 8 KB, 1024-byte aligned).
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * 8192) + sw128_offset(row, chunk & 7);
}

template <int D>
struct WarpAttn {
  float o[D / 8][4];  // O~ fragments: rows g, g+8 (g = lane/4), columns 8n + 2(lane%4) + {0,1}
  float m[2];         // running max, base-2 units, rows g and g+8 (equal across the quad)
  float l[2];         // this thread's partial row sums
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m[0] = m[1] = neg_inf();
    l[0] = l[1] = 0.f;
  }
  // full row sums (quad reduction)
  __device__ __forceinline__ void reduce_l() {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
    }
  }
};

// A fragments of 16 query rows (row0..row0+15) for all D/16 k-steps.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][4], uint32_t q_tile, int row0, int lane) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) ldmatrix_x4(qf[kk], q_tile + tile_off(row0 + (lane & 15), 2 * kk + (lane >> 4)));
}

// One online-softmax step (LaCache Eq. (2)-(6)) of a warp's 16 rows with the
// NK keys key0..key0+NK-1 of a K/V tile pair; key j takes part iff valid(j).
// FRESH: st is the empty state (m = -inf, l = 0, O~ = 0), so nothing is rescaled.
template <int D, int NK, bool FRESH = false, class Valid>
__device__ __forceinline__ void attend(WarpAttn<D>& st, const uint32_t (&qf)[D / 16][4], uint32_t k_tile,
                                       uint32_t v_tile, int key0, float scale_log2, Valid valid, int lane) {
  float s[NK / 8][4];
#pragma unroll
  for (int n = 0; n < NK / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
  // S = Q K^T
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int jn = 0; jn < NK / 16; ++jn) {
      uint32_t b[4];
      ldmatrix_x4(b, k_tile + tile_off(key0 + jn * 16 + (lane & 7) + ((lane >> 4) << 3), 2 * kk + ((lane >> 3) & 1)));
      const uint32_t b01[2] = {b[0], b[1]}, b23[2] = {b[2], b[3]};
      mma_bf16_16816(s[2 * jn], qf[kk], b01);
      mma_bf16_16816(s[2 * jn + 1], qf[kk], b23);
    }
  }
  // scale, mask, row max (Eq. (2))
  const int t = lane & 3;
  float mx0 = neg_inf(), mx1 = neg_inf();
#pragma unroll
  for (int n = 0; n < NK / 8; ++n) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const bool ok = valid(key0 + n * 8 + 2 * t + e);
      s[n][e] = ok ? s[n][e] * scale_log2 : neg_inf();
      s[n][2 + e] = ok ? s[n][2 + e] * scale_log2 : neg_inf();
      mx0 = fmaxf(mx0, s[n][e]);
      mx1 = fmaxf(mx1, s[n][2 + e]);
    }
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = FRESH ? mx0 : fmaxf(st.m[0], mx0), mn1 = FRESH ? mx1 : fmaxf(st.m[1], mx1);
  const float mu0 = mn0 == neg_inf() ? 0.f : mn0, mu1 = mn1 == neg_inf() ? 0.f : mn1;
  const float a0 = FRESH ? 0.f : fast_exp2(st.m[0] - mu0);  // Eq. (3); empty state -> 0
  const float a1 = FRESH ? 0.f : fast_exp2(st.m[1] - mu1);
  st.m[0] = mn0;
  st.m[1] = mn1;
  float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
  for (int n = 0; n < NK / 8; ++n) {  // Eq. (4)
    s[n][0] = fast_exp2(s[n][0] - mu0);
    s[n][1] = fast_exp2(s[n][1] - mu0);
    s[n][2] = fast_exp2(s[n][2] - mu1);
    s[n][3] = fast_exp2(s[n][3] - mu1);
    rs0 += s[n][0] + s[n][1];
    rs1 += s[n][2] + s[n][3];
  }
  st.l[0] = FRESH ? rs0 : st.l[0] * a0 + rs0;  // Eq. (5), per-thread partial
  st.l[1] = FRESH ? rs1 : st.l[1] * a1 + rs1;
  if (!FRESH) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {  // Eq. (6), first term
      st.o[n][0] *= a0;
      st.o[n][1] *= a0;
      st.o[n][2] *= a1;
      st.o[n][3] *= a1;
    }
  }
  // Eq. (6), second term: O~ += P V
#pragma unroll
  for (int kk = 0; kk < NK / 16; ++kk) {
    const uint32_t pa[4] = {pack_bf16x2(s[2 * kk][0], s[2 * kk][1]), pack_bf16x2(s[2 * kk][2], s[2 * kk][3]),
                            pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                            pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn) {
      uint32_t b[4];
      ldmatrix_x4_trans(b, v_tile + tile_off(key0 + kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                             2 * dn + (lane >> 4)));
      const uint32_t b01[2] = {b[0], b[1]}, b23[2] = {b[2], b[3]};
      if (FRESH && kk == 0) {  // the first product over the empty state: C = 0
        mma_bf16_16816_zc(st.o[2 * dn], pa, b01);
        mma_bf16_16816_zc(st.o[2 * dn + 1], pa, b23);
      } else {
        mma_bf16_16816(st.o[2 * dn], pa, b01);
        mma_bf16_16816(st.o[2 * dn + 1], pa, b23);
      }
    }
  }
}

// Per-sequence metadata, validated against the host bounds.
struct SeqMeta {
  int nb, bb, sb, cub, cus;
  bool ok;
};

__device__ __forceinline__ SeqMeta load_meta(const BatchArgs& bt, int b) {
  SeqMeta m;
  m.nb = __ldg(bt.seq_len + b);
  m.bb = __ldg(bt.block_len + b);
  m.sb = __ldg(bt.block_start + b);
  m.cub = __ldg(bt.cu_block + b);
  m.cus = __ldg(bt.cu_seq + b);
  m.ok = m.nb >= 1 && m.nb <= bt.max_seq_len && m.bb >= 1 && m.bb <= bt.max_block_len && m.bb <= 64 &&
         m.sb >= 0 && m.sb + m.bb <= m.nb && (m.nb + kPage - 1) / kPage <= bt.max_pages && m.cub >= 0 &&
         m.cub + m.bb <= bt.total_block_rows && m.cus >= 0 && m.cus + m.nb <= bt.total_seq_rows;
  return m;
}

// A block-table entry in two steps, so that its load can be issued well before its use:
// page_raw loads it, page_checked validates it.
__device__ __forceinline__ int page_raw(const BatchArgs& bt, int b, int p) {
  return __ldg(bt.block_table + static_cast<size_t>(b) * bt.max_pages + p);
}
__device__ __forceinline__ int page_checked(const BatchArgs& bt, int pg) {
  if (pg < 0 || pg >= bt.num_pages) {
    report_error(bt.err, kErrBadPage);
    pg = 0;  // load an in-bounds page; the result is flagged as invalid
  }
  return pg;
}
__device__ __forceinline__ int page_of(const BatchArgs& bt, int b, int p) { return page_checked(bt, page_raw(bt, b, p)); }

template <int D>
constexpr int tile_bytes() {
  return (D / 64) * 8192;
}

// ------------------------------------------------------------ launch helpers
template <class K>
cudaError_t set_smem(K kern, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)  // all of the unified L1/shared storage as shared memory: more resident CTAs
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  return e;
}

// Launch with programmatic stream serialization (and an optional cluster shape).
template <class K, class... Args>
cudaError_t launch_pdl(K kern, dim3 grid, int threads, int smem, int cluster_x, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster_x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct PoolMaps {
  CUtensorMap k, v, q, o;
};

inline cudaError_t encode_pool_maps(const AttnArgs& a, bool need_q, bool need_o, PoolMaps* m) {
  const uint64_t rows = static_cast<uint64_t>(a.bt.num_pages) * a.n_heads * kPage;
  const uint64_t d = a.head_dim;
  cudaError_t e = encode_2d_sw128(&m->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k_pool, d, rows, 64, 64);
  if (e == cudaSuccess) e = encode_2d_sw128(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v_pool, d, rows, 64, 64);
  if (e == cudaSuccess && need_q)
    e = encode_2d_sw128(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_pool, d, rows, 64, 64);
  if (e == cudaSuccess && need_o)
    e = encode_2d_sw128(&m->o, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.o_pool, d, rows, 64, 64);
  return e;
}

}  // namespace attn
}  // namespace dllm
