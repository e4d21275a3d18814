// attention.cu — the FACache build of a block boundary (sm_103a).
//
//   state_build_kernel   per row of U, the online-softmax state (m, l, O~)
//                        over the keys of U only (LaCache §3.3.3; Algorithm 1
//                        with GenStep = True).
//
// One CTA per (query page, head, sequence): a producer warp streams the
// query page and every 64-token K/V page of the sequence with TMA (128-byte
// swizzle) into an mbarrier ring; 4 warps run QK^T / PV of their 16 query
// rows on mma.sync m16n8k16 with keys of C masked out.  The block attention
// and the FACache merge of the inner steps are in attn_stream.cu.
#include "attn_common.cuh"

namespace dllm {
namespace {
using namespace attn;

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

}  // namespace

namespace {
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

}  // namespace

cudaError_t launch_state_build(const AttnArgs& a, cudaStream_t stream) {
  if (a.bt.batch <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_state_build_d<128>(a, stream) : launch_state_build_d<64>(a, stream);
}

}  // namespace dllm
