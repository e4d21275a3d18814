// attention.cu — the three attention kernels of the step (sm_103a):
//
//   block_attention_kernel  block rows (<= 64 queries of one sequence and
//                           head) over every key of the sequence, read page
//                           by page through the block table (Fast-dLLM
//                           DualCache: [prefix KV | fresh block KV | suffix KV]).
//   state_build_kernel      FACache build: per row of U, the online-softmax
//                           state (m, l, O~) over the keys of U only
//                           (LaCache §3.3.3; Algorithm 1 with GenStep = True).
//   state_merge_kernel      FACache reuse: per row of U, the cached state
//                           merged with the fresh block keys (LaCache Eq.
//                           (2)-(6); Algorithm 1 with GenStep = False).
//
// All three stream 64-token pages of bf16 K/V (and Q, O~) with TMA tile
// loads (128-byte swizzle, so the ldmatrix reads below are bank-conflict
// free) into an mbarrier ring filled by a producer warp, and run the
// QK^T / PV contractions of each warp's 16 query rows on the warp-level
// tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate).  These contractions
// are tiny (<= 64 queries) and bandwidth-bound; row max and row sum use quad
// shuffles.  The online softmax works in base 2: scores are pre-multiplied
// by scale * log2(e) and every m kept on chip is in those units; the ABI's
// m_pool and lse are natural-log units.
//
// Block attention splits the pages of a (sequence, head) across the CTAs of
// a thread-block cluster; the partial states are combined exactly (the same
// Eq. (2)-(6) merge) through distributed shared memory, so no partial ever
// reaches HBM.  Each CTA pushes its combined partial of row i into the
// shared memory of the CTA that owns row i (i mod cluster size) with remote
// 16-byte stores, so the exchange costs one store per element and two
// cluster barriers; the owners then finish their rows from local memory.
//
// All three kernels are launched with programmatic dependent launch: barrier
// setup overlaps the tail of the preceding kernel, and every read of data a
// preceding kernel may write comes after griddepcontrol.wait.
#include "kernels.cuh"
#include "sm103.cuh"
#include "tmap.cuh"

namespace dllm {
namespace {

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
template <int D, int NK, class Valid>
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
  const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
  const float mu0 = mn0 == neg_inf() ? 0.f : mn0, mu1 = mn1 == neg_inf() ? 0.f : mn1;
  const float a0 = fast_exp2(st.m[0] - mu0), a1 = fast_exp2(st.m[1] - mu1);  // Eq. (3); empty state -> 0
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
  st.l[0] = st.l[0] * a0 + rs0;  // Eq. (5), per-thread partial
  st.l[1] = st.l[1] * a1 + rs1;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {  // Eq. (6), first term
    st.o[n][0] *= a0;
    st.o[n][1] *= a0;
    st.o[n][2] *= a1;
    st.o[n][3] *= a1;
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
      mma_bf16_16816(st.o[2 * dn], pa, b01);
      mma_bf16_16816(st.o[2 * dn + 1], pa, b23);
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

__device__ __forceinline__ int page_of(const BatchArgs& bt, int b, int p) {
  int pg = __ldg(bt.block_table + static_cast<size_t>(b) * bt.max_pages + p);
  if (pg < 0 || pg >= bt.num_pages) {
    report_error(bt.err, kErrBadPage);
    pg = 0;  // load an in-bounds page; the result is flagged as invalid
  }
  return pg;
}

template <int D>
constexpr int tile_bytes() {
  return (D / 64) * 8192;
}

// ========================================================= block attention
template <int D>
struct BlockAttnCfg {
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kSmem = tile_bytes<D>() * (1 + 2 * kStages) + 1024;
  static constexpr int kOStride = D + 8;  // padded fp32 row of the per-warp partials
  static constexpr int kCombBytes = 64 * kOStride * 4;
  // Receive slots of the owner CTA: D accumulator floats, then (m, l) and
  // padding; rows i = rank + S*il, slot il*S + r for peer r (< 72 slots).
  static constexpr int kRecvStride = D + 4;
  static constexpr int kRecvSlots = 72;
  static_assert(kCombBytes + kRecvSlots * kRecvStride * 4 <= tile_bytes<D>() * (1 + 2 * kStages),
                "combine buffers must fit in the q tile and the drained ring");
};

template <int D>
__global__ void __launch_bounds__(160) block_attention_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                              const __grid_constant__ CUtensorMap tm_v,
                                                              const AttnArgs a) {
  constexpr int TB = tile_bytes<D>();
  constexpr int NST = BlockAttnCfg<D>::kStages;
  constexpr int OS = BlockAttnCfg<D>::kOStride;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  constexpr int RS = BlockAttnCfg<D>::kRecvStride;
  uint8_t* q_tile = smem;
  uint8_t* kv = smem + TB;
  // After the page loop the q tile and the ring hold the combine buffers.
  float* comb_o = reinterpret_cast<float*>(smem);  // [64][OS] per-warp partials of this CTA
  float* recv = reinterpret_cast<float*>(smem + BlockAttnCfg<D>::kCombBytes);  // [72][RS] pushed partials
  __shared__ uint64_t full_bar[NST], empty_bar[NST];
  __shared__ float comb_m[64], comb_l[64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y, rank = blockIdx.x, S = gridDim.x;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  griddep_wait();  // q_block, the pools (and any metadata) may come from the preceding kernel
  SeqMeta sm = load_meta(bt, b);
  if (!sm.ok) {
    if (threadIdx.x == 0 && rank == 0 && h == 0) report_error(bt.err, kErrBadShape);
    sm.nb = 0;
    sm.bb = 0;
  }
  const int npages = (sm.nb + kPage - 1) / kPage;
  const int ppc = (npages + S - 1) / S;
  const int p0 = min(npages, rank * ppc), p1 = min(npages, p0 + ppc);
  const int my = p1 - p0;
  const int RG = (sm.bb + 15) / 16;    // 16-row groups of block queries
  const int KS = RG > 0 ? 4 / RG : 1;  // key slices per page
  const bool active = warp < 4 && RG > 0 && warp < RG * KS;
  const int rg = RG > 0 ? warp % RG : 0, ks = RG > 0 ? warp / RG : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 4);
    }
    fence_barrier_init();
  }
  if (warp < 4) {  // queries of the block rows, zero-padded to 64 rows
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q_block);
    for (int e = threadIdx.x; e < 64 * (D / 8); e += 128) {
      const int row = e / (D / 8), ch = e % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < sm.bb)
        v = __ldg(reinterpret_cast<const uint4*>(qb + (static_cast<size_t>(sm.cub + row) * H + h) * D) + ch);
      *reinterpret_cast<uint4*>(q_tile + tile_off(row, ch)) = v;
    }
  }
  __syncthreads();

  WarpAttn<D> st;
  st.init();
  if (warp == 4) {
    if (lane == 0) {  // ---- TMA producer
      int issued = 0;
      for (int i = 0; i < my; ++i) {
        const int s = i % NST;
        const uint32_t ph = (i / NST) & 1;
        if (i >= NST && !mbar_wait(&empty_bar[s], ph ^ 1)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        const int pg = page_of(bt, b, p0 + i);
        uint8_t* kt = kv + s * 2 * TB;
        const int y = (pg * H + h) * kPage;
        mbar_arrive_expect_tx(&full_bar[s], 2 * TB);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_2d(kt + hf * 8192, &tm_k, &full_bar[s], hf * 64, y);
          tma_load_2d(kt + TB + hf * 8192, &tm_v, &full_bar[s], hf * 64, y);
        }
        ++issued;
      }
      for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % NST], (i / NST) & 1)) report_error(bt.err, kErrTimeout);
    }
  } else {  // ---- compute warps
    uint32_t qf[D / 16][4];
    if (active) load_q_frags<D>(qf, smem_u32(q_tile), rg * 16, lane);
    const int nk = 64 / KS, key0 = ks * nk;
    for (int i = 0; i < my; ++i) {
      const int s = i % NST;
      const uint32_t ph = (i / NST) & 1;
      if (!mbar_wait(&full_bar[s], ph)) {
        report_error(bt.err, kErrTimeout);
        break;
      }
      if (active) {
        const uint32_t kt = smem_u32(kv + s * 2 * TB), vt = kt + TB;
        const int base = (p0 + i) * kPage;
        const int nb = sm.nb;
        auto valid = [base, nb](int key) { return base + key < nb; };
        if (KS == 1)
          attend<D, 64>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
        else if (KS == 2)
          attend<D, 32>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
        else
          attend<D, 16>(st, qf, kt, vt, key0, a.scale_log2, valid, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
  }
  __syncthreads();  // every page consumed and every load landed: the ring becomes the combine buffer
  // Peers may push into this CTA's receive slots once every CTA of the
  // cluster is past its page loop.
  cluster_arrive_release();

  if (active) {
    st.reduce_l();
    const int g = lane >> 2, t = lane & 3;
    const int slot0 = ks * RG * 16 + rg * 16 + g, slot1 = slot0 + 8;
    if (t == 0) {
      comb_m[slot0] = st.m[0];
      comb_l[slot0] = st.l[0];
      comb_m[slot1] = st.m[1];
      comb_l[slot1] = st.l[1];
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      *reinterpret_cast<float2*>(comb_o + slot0 * OS + 8 * n + 2 * t) = make_float2(st.o[n][0], st.o[n][1]);
      *reinterpret_cast<float2*>(comb_o + slot1 * OS + 8 * n + 2 * t) = make_float2(st.o[n][2], st.o[n][3]);
    }
  }
  __syncthreads();
  cluster_wait_acquire();

  // ---- combine the KS key-slice partials of each block row (Eq. (2)-(6)
  // applied to states) and push the result to the row's owner i % S
  constexpr int C4 = D / 4;
  const uint32_t recv_addr = smem_u32(recv);
  for (int item = threadIdx.x; item < sm.bb * C4; item += 160) {
    const int i = item / C4, c = (item % C4) * 4;
    float M = neg_inf();
    for (int q = 0; q < KS; ++q) M = fmaxf(M, comb_m[q * RG * 16 + i]);
    const float Mu = M == neg_inf() ? 0.f : M;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < KS; ++q) {
      const int slot = q * RG * 16 + i;
      const float w = fast_exp2(comb_m[slot] - Mu);
      L += w * comb_l[slot];
      const float4 ov = *reinterpret_cast<const float4*>(comb_o + slot * OS + c);
      acc.x += w * ov.x;
      acc.y += w * ov.y;
      acc.z += w * ov.z;
      acc.w += w * ov.w;
    }
    const int owner = i % S, rslot = (i / S) * S + rank;
    const uint32_t dst = mapa_shared(recv_addr + static_cast<uint32_t>((rslot * RS + c) * 4), owner);
    st_shared_cluster_v4(dst, acc);
    if (c == 0)
      st_shared_cluster_v4(mapa_shared(recv_addr + static_cast<uint32_t>((rslot * RS + D) * 4), owner),
                           make_float4(M, L, 0.f, 0.f));
  }
  cluster_arrive_release();  // pushes are visible to their owners after the wait
  cluster_wait_acquire();
  griddep_launch_dependents();

  // ---- the owner merges the S pushed partials of its rows i = rank + S*il
  {
    const int nmine = sm.bb > rank ? (sm.bb - rank + S - 1) / S : 0;
    __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
    for (int item = threadIdx.x; item < nmine * C4; item += 160) {
      const int il = item / C4, c = (item % C4) * 4;
      const int i = rank + S * il;
      const float* base = recv + il * S * RS;
      float M = neg_inf();
      for (int r = 0; r < S; ++r) M = fmaxf(M, base[r * RS + D]);
      const float Mu = M == neg_inf() ? 0.f : M;
      float L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < S; ++r) {
        const float* pr = base + r * RS;
        const float w = fast_exp2(pr[D] - Mu);
        L += w * pr[D + 1];
        const float4 ov = *reinterpret_cast<const float4*>(pr + c);
        acc.x += w * ov.x;
        acc.y += w * ov.y;
        acc.z += w * ov.z;
        acc.w += w * ov.w;
      }
      const float inv = 1.f / L;
      const size_t orow = static_cast<size_t>(sm.cus + sm.sb + i) * H + h;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(of + orow * D + c) = pk;
      if (a.lse != nullptr && c == 0) a.lse[orow] = (M + log2f(L)) * kLn2;
    }
  }
}

// ============================================================= state build
template <int D>
struct StateBuildCfg {
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kSmem = tile_bytes<D>() * (1 + 2 * kStages) + 1024;
};

template <int D>
__global__ void __launch_bounds__(160) state_build_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                          const __grid_constant__ CUtensorMap tm_k,
                                                          const __grid_constant__ CUtensorMap tm_v,
                                                          const AttnArgs a) {
  constexpr int TB = tile_bytes<D>();
  constexpr int NST = StateBuildCfg<D>::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* q_tile = smem;
  uint8_t* kv = smem + TB;
  __shared__ uint64_t full_bar[NST], empty_bar[NST], q_bar;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  griddep_wait();  // the pools (and any metadata) may come from the preceding kernel
  griddep_launch_dependents();
  const SeqMeta sm = load_meta(bt, b);
  if (!sm.ok) {
    if (threadIdx.x == 0 && qp == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int npages = (sm.nb + kPage - 1) / kPage;
  if (qp >= npages) return;
  // rows of this page that belong to U
  const int r_lo = qp * kPage, r_hi = min(sm.nb, r_lo + kPage);
  const bool has_u = (r_lo < sm.sb) || (r_hi > sm.sb + sm.bb);
  if (!has_u) return;
  const int pgq = page_of(bt, b, qp);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 4);
    }
    mbar_init(&q_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  WarpAttn<D> st;
  st.init();
  if (warp == 4) {
    if (lane == 0) {  // ---- TMA producer: the query page, then every key page
      mbar_arrive_expect_tx(&q_bar, TB);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(q_tile + hf * 8192, &tm_q, &q_bar, hf * 64, (pgq * H + h) * kPage);
      int issued = 0;
      for (int i = 0; i < npages; ++i) {
        const int s = i % NST;
        const uint32_t ph = (i / NST) & 1;
        if (i >= NST && !mbar_wait(&empty_bar[s], ph ^ 1)) {
          report_error(bt.err, kErrTimeout);
          break;
        }
        const int pg = page_of(bt, b, i);
        uint8_t* kt = kv + s * 2 * TB;
        const int y = (pg * H + h) * kPage;
        mbar_arrive_expect_tx(&full_bar[s], 2 * TB);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_2d(kt + hf * 8192, &tm_k, &full_bar[s], hf * 64, y);
          tma_load_2d(kt + TB + hf * 8192, &tm_v, &full_bar[s], hf * 64, y);
        }
        ++issued;
      }
      for (int i = (issued > NST ? issued - NST : 0); i < issued; ++i)
        if (!mbar_wait(&full_bar[i % NST], (i / NST) & 1)) report_error(bt.err, kErrTimeout);
      if (!mbar_wait(&q_bar, 0)) report_error(bt.err, kErrTimeout);
    }
  } else {
    uint32_t qf[D / 16][4];
    const bool q_ok = mbar_wait(&q_bar, 0);
    if (!q_ok) report_error(bt.err, kErrTimeout);
    load_q_frags<D>(qf, smem_u32(q_tile), warp * 16, lane);
    const int nb = sm.nb, c_lo = sm.sb, c_hi = sm.sb + sm.bb;
    for (int i = 0; i < npages && q_ok; ++i) {
      const int s = i % NST;
      const uint32_t ph = (i / NST) & 1;
      if (!mbar_wait(&full_bar[s], ph)) {
        report_error(bt.err, kErrTimeout);
        break;
      }
      const uint32_t kt = smem_u32(kv + s * 2 * TB), vt = kt + TB;
      const int base = i * kPage;
      auto valid = [base, nb, c_lo, c_hi](int key) {
        const int p = base + key;
        return p < nb && (p < c_lo || p >= c_hi);  // keys of U only
      };
      attend<D, 64>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }
    // ---- store the state of the U rows of this page
    st.reduce_l();
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = warp * 16 + g + 8 * hr;
      const int pos = r_lo + r;
      if (pos >= sm.nb || (pos >= c_lo && pos < c_hi)) continue;
      const size_t srow = (static_cast<size_t>(pgq) * H + h) * kPage + r;
      if (t == 0) {
        a.m_pool[srow] = st.m[hr] * kLn2;  // natural units; -inf stays -inf
        a.l_pool[srow] = st.l[hr];
      }
      float* orow = a.o_pool + srow * D;
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(orow + 8 * n + 2 * t) = make_float2(st.o[n][2 * hr], st.o[n][2 * hr + 1]);
    }
  }
}

// ============================================================= state merge
template <int D>
struct MergeCfg {
  // q tile | K_C | V_C | O~ tile (fp32: D/32 swizzled boxes of 32 columns x 64 rows)
  static constexpr int kSmem = tile_bytes<D>() * 3 + 64 * D * 4 + 1024;
};

template <int D>
__global__ void __launch_bounds__(128) state_merge_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                          const __grid_constant__ CUtensorMap tm_o,
                                                          const AttnArgs a) {
  constexpr int TB = tile_bytes<D>();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* q_tile = smem;       // later: staging of the bf16 output rows
  uint8_t* kc_tile = smem + TB;
  uint8_t* vc_tile = smem + 2 * TB;
  uint8_t* o_tile = smem + 3 * TB;
  __shared__ uint64_t t_bar;
  __shared__ float m_s[64], l_s[64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const BatchArgs& bt = a.bt;
  const int H = a.n_heads;
  griddep_wait();  // the fresh block keys (and any metadata) may come from the preceding kernel
  griddep_launch_dependents();
  const SeqMeta sm = load_meta(bt, b);
  if (!sm.ok) {
    if (threadIdx.x == 0 && qp == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int npages = (sm.nb + kPage - 1) / kPage;
  if (qp >= npages) return;
  const int r_lo = qp * kPage, r_hi = min(sm.nb, r_lo + kPage);
  const int c_lo = sm.sb, c_hi = sm.sb + sm.bb;
  if (!((r_lo < c_lo) || (r_hi > c_hi))) return;  // no row of U in this page
  const int pgq = page_of(bt, b, qp);
  const size_t srow0 = (static_cast<size_t>(pgq) * H + h) * kPage;

  if (threadIdx.x == 0) {
    mbar_init(&t_bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // queries and cached O~ of the page's rows
    mbar_arrive_expect_tx(&t_bar, TB + 64 * D * 4);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) tma_load_2d(q_tile + hf * 8192, &tm_q, &t_bar, hf * 64, static_cast<int>(srow0));
#pragma unroll
    for (int j = 0; j < D / 32; ++j) tma_load_2d(o_tile + j * 8192, &tm_o, &t_bar, j * 32, static_cast<int>(srow0));
  }
  // cached m, l of the page's rows; block keys/values gathered through the table
  if (threadIdx.x < 64) {
    m_s[threadIdx.x] = a.m_pool[srow0 + threadIdx.x];
    l_s[threadIdx.x] = a.l_pool[srow0 + threadIdx.x];
  }
  const int nkc = (sm.bb + 15) & ~15;
  {
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(a.k_pool);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(a.v_pool);
    for (int e = threadIdx.x; e < nkc * (D / 8); e += 128) {
      const int c = e / (D / 8), ch = e % (D / 8);
      uint4 kv4 = make_uint4(0, 0, 0, 0), vv4 = make_uint4(0, 0, 0, 0);
      if (c < sm.bb) {
        const int pos = c_lo + c;
        const int pg = page_of(bt, b, pos / kPage);
        const size_t off = ((static_cast<size_t>(pg) * H + h) * kPage + (pos % kPage)) * D;
        kv4 = __ldg(reinterpret_cast<const uint4*>(kp + off) + ch);
        vv4 = __ldg(reinterpret_cast<const uint4*>(vp + off) + ch);
      }
      *reinterpret_cast<uint4*>(kc_tile + tile_off(c, ch)) = kv4;
      *reinterpret_cast<uint4*>(vc_tile + tile_off(c, ch)) = vv4;
    }
  }
  __syncthreads();
  const bool loaded = mbar_wait(&t_bar, 0);
  if (!loaded) report_error(bt.err, kErrTimeout);

  // fresh partial state over the block keys (Eq. (2)-(6) from the empty state)
  WarpAttn<D> st;
  st.init();
  uint32_t qf[D / 16][4];
  load_q_frags<D>(qf, smem_u32(q_tile), warp * 16, lane);
  const uint32_t kt = smem_u32(kc_tile), vt = smem_u32(vc_tile);
  const int bb = sm.bb;
  auto valid = [bb](int key) { return key < bb; };
  if (nkc == 16)
    attend<D, 16>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else if (nkc == 32)
    attend<D, 32>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else if (nkc == 48)
    attend<D, 48>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  else
    attend<D, 64>(st, qf, kt, vt, 0, a.scale_log2, valid, lane);
  st.reduce_l();

  // exact merge with the cached state, staged as bf16 rows in the q tile
  const int g = lane >> 2, t = lane & 3;
  const float log2e = 1.4426950408889634f;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = warp * 16 + g + 8 * hr;
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
    if (a.lse != nullptr && t == 0 && pos < sm.nb && (pos < c_lo || pos >= c_hi))
      a.lse[static_cast<size_t>(sm.cus + pos) * H + h] = (M + log2f(L)) * kLn2;
  }
  __syncwarp();
  // coalesced store of this warp's 16 rows
  __nv_bfloat16* of = static_cast<__nv_bfloat16*>(a.o_full);
  for (int e = lane; e < 16 * (D / 8); e += 32) {
    const int r = warp * 16 + e / (D / 8), ch = e % (D / 8);
    const int pos = r_lo + r;
    if (pos >= sm.nb || (pos >= c_lo && pos < c_hi)) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(q_tile + tile_off(r, ch));
    *reinterpret_cast<uint4*>(of + (static_cast<size_t>(sm.cus + pos) * H + h) * D + ch * 8) = v;
  }
}

// ================================================================ launchers
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

cudaError_t encode_pool_maps(const AttnArgs& a, bool need_q, bool need_o, PoolMaps* m) {
  const uint64_t rows = static_cast<uint64_t>(a.bt.num_pages) * a.n_heads * kPage;
  const uint64_t d = a.head_dim;
  cudaError_t e = encode_2d_sw128(&m->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.k_pool, d, rows, 64, 64);
  if (e == cudaSuccess) e = encode_2d_sw128(&m->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.v_pool, d, rows, 64, 64);
  if (e == cudaSuccess && need_q)
    e = encode_2d_sw128(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q_pool, d, rows, 64, 64);
  if (e == cudaSuccess && need_o)
    e = encode_2d_sw128(&m->o, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.o_pool, d, rows, 32, 64);
  return e;
}

template <int D>
cudaError_t launch_block_attention_d(const AttnArgs& a, int num_sms, cudaStream_t stream) {
  PoolMaps m;
  cudaError_t e = encode_pool_maps(a, false, false, &m);
  if (e != cudaSuccess) return e;
  constexpr int smem = BlockAttnCfg<D>::kSmem;
  auto kern = block_attention_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  // Split each (sequence, head) over a cluster of S CTAs so that the grid
  // covers the SMs about twice; at most 8 (portable cluster size) and at
  // most one CTA per page.
  const long long units = static_cast<long long>(a.bt.batch) * a.n_heads;
  const int max_pages = (a.bt.max_seq_len + kPage - 1) / kPage;
  int split = static_cast<int>((2LL * num_sms + units - 1) / units);
  if (split > 8) split = 8;
  if (split > max_pages) split = max_pages;
  if (split < 1) split = 1;
  return launch_pdl(kern, dim3(split, a.n_heads, a.bt.batch), 160, smem, split, stream, m.k, m.v, a);
}

template <int D>
cudaError_t launch_state_build_d(const AttnArgs& a, cudaStream_t stream) {
  PoolMaps m;
  cudaError_t e = encode_pool_maps(a, true, false, &m);
  if (e != cudaSuccess) return e;
  constexpr int smem = StateBuildCfg<D>::kSmem;
  auto kern = state_build_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int max_pages = (a.bt.max_seq_len + kPage - 1) / kPage;
  return launch_pdl(kern, dim3(max_pages, a.n_heads, a.bt.batch), 160, smem, 0, stream, m.q, m.k, m.v, a);
}

template <int D>
cudaError_t launch_state_merge_d(const AttnArgs& a, cudaStream_t stream) {
  PoolMaps m;
  cudaError_t e = encode_pool_maps(a, true, true, &m);
  if (e != cudaSuccess) return e;
  constexpr int smem = MergeCfg<D>::kSmem;
  auto kern = state_merge_kernel<D>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int max_pages = (a.bt.max_seq_len + kPage - 1) / kPage;
  return launch_pdl(kern, dim3(max_pages, a.n_heads, a.bt.batch), 128, smem, 0, stream, m.q, m.o, a);
}

}  // namespace

cudaError_t launch_block_attention(const AttnArgs& a, int num_sms, cudaStream_t stream) {
  if (a.bt.batch <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_block_attention_d<128>(a, num_sms, stream)
                           : launch_block_attention_d<64>(a, num_sms, stream);
}

cudaError_t launch_state_build(const AttnArgs& a, cudaStream_t stream) {
  if (a.bt.batch <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_state_build_d<128>(a, stream) : launch_state_build_d<64>(a, stream);
}

cudaError_t launch_state_merge(const AttnArgs& a, cudaStream_t stream) {
  if (a.bt.batch <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_state_merge_d<128>(a, stream) : launch_state_merge_d<64>(a, stream);
}

}  // namespace dllm
