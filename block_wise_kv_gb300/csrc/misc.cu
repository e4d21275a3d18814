// misc.cu — the small kernels around the projection:
//   * the RoPE cos/sin table (LaCache Eq. (1), rotate-half pairs),
//   * zeroing of the pool slots past the end of each sequence, so that the
//     attention kernels may load whole 64-token pages.
#include "kernels.cuh"
#include "sm103.cuh"

namespace dllm {
namespace {

// table[p][i] = (cos, sin)(p * theta^(-2i/d)), angle and trig in fp64.
__global__ void rope_table_kernel(float* __restrict__ table, int max_pos, int head_dim, double theta) {
  const int half = head_dim / 2;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(max_pos) * half) return;
  const int p = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
  const double inv_freq = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(head_dim));
  double s, c;
  sincos(static_cast<double>(p) * inv_freq, &s, &c);
  table[2 * idx] = static_cast<float>(c);
  table[2 * idx + 1] = static_cast<float>(s);
}

// Grid (batch, heads): zero slots [N_b, 64 * ceil(N_b / 64)) of the last page
// of sequence b in the k, v and q pools.
__global__ void zero_tails_kernel(BatchArgs bt, __nv_bfloat16* k_pool, __nv_bfloat16* v_pool,
                                  __nv_bfloat16* q_pool, int H, int d) {
  const int b = blockIdx.x, h = blockIdx.y;
  const int nb = bt.seq_len[b];
  if (nb < 1 || nb > bt.max_seq_len) {
    if (threadIdx.x == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int np = (nb + kPage - 1) / kPage;
  const int first = nb - (np - 1) * kPage;  // live slots in the last page
  if (first == kPage) return;
  if (np > bt.max_pages) {
    if (threadIdx.x == 0 && h == 0) report_error(bt.err, kErrBadShape);
    return;
  }
  const int pg = bt.block_table[static_cast<size_t>(b) * bt.max_pages + np - 1];
  if (pg < 0 || pg >= bt.num_pages) {
    if (threadIdx.x == 0 && h == 0) report_error(bt.err, kErrBadPage);
    return;
  }
  const int vec_per_row = d / 8;
  const int nvec = (kPage - first) * vec_per_row;
  const size_t base = ((static_cast<size_t>(pg) * H + h) * kPage + first) * d;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    reinterpret_cast<uint4*>(k_pool + base)[v] = z;
    reinterpret_cast<uint4*>(v_pool + base)[v] = z;
    reinterpret_cast<uint4*>(q_pool + base)[v] = z;
  }
}

}  // namespace

cudaError_t launch_rope_table(float* table, int max_pos, int head_dim, double theta, cudaStream_t stream) {
  const long long n = static_cast<long long>(max_pos) * (head_dim / 2);
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  rope_table_kernel<<<static_cast<unsigned>((n + threads - 1) / threads), threads, 0, stream>>>(table, max_pos,
                                                                                                head_dim, theta);
  return cudaGetLastError();
}

cudaError_t launch_zero_tails(const BatchArgs& bt, void* k_pool, void* v_pool, void* q_pool, int n_heads,
                              int head_dim, cudaStream_t stream) {
  if (bt.batch <= 0) return cudaSuccess;
  zero_tails_kernel<<<dim3(bt.batch, n_heads), 128, 0, stream>>>(
      bt, static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool),
      static_cast<__nv_bfloat16*>(q_pool), n_heads, head_dim);
  return cudaGetLastError();
}

}  // namespace dllm
