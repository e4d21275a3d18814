// misc.cu — the small kernels around the projection:
//   * RMSNorm of token rows into the bf16 operand of the projection
//     (LaCache §3.3.2: the attention norm is a token-wise operator),
//   * the RoPE cos/sin table (LaCache Eq. (1), rotate-half pairs),
//   * zeroing of the pool slots past the end of each sequence, so that the
//     attention kernels may load whole 64-token pages.
#include "kernels.cuh"
#include "sm103.cuh"

namespace dllm {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormVecs = 4;  // 16-byte vectors of the row kept in registers per thread (D <= 8192)

// s + e == a + b exactly (Knuth's TwoSum), with the additions pinned to
// round-to-nearest so that the compiler cannot contract or reorder them.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// bf16 nearest-even rounding of the real value p + e, where p = fl32(p + e)
// and |e| is below half an fp32 step of p: p alone decides unless p sits
// exactly on a bf16 midpoint, in which case the sign of e does.
__device__ __forceinline__ uint16_t bf16_round_pair(float p, float e) {
  const uint32_t bits = __float_as_uint(p);
  if ((bits & 0xFFFFu) == 0x8000u && e != 0.f) {
    const bool away = (e > 0.f) == (p > 0.f);
    return static_cast<uint16_t>((bits >> 16) + (away ? 1u : 0u));
  }
  return __bfloat16_as_ushort(__float2bfloat16_rn(p));
}

// 1 / sqrt(ss / D + eps) as an unevaluated pair (hi, lo) of floats, from the
// exact sum of squares (ss_hi, ss_lo), in fp32 arithmetic only (fp64 is slow
// on this part).  The quotient and the sum are carried as float pairs
// (the division remainder by FMA is exact); the reciprocal square root is
// one Newton-Raphson step y1 = y0 - y0 (s y0^2 - 1) / 2 from the hardware
// estimate y0 (relative error e0 < 2^-21), with the residual s y0^2 - 1
// formed from an exact product y0^2 and FMAs.  Newton's error (3/2) e0^2 and
// the rounding of the residual leave |y1 / y - 1| below about 2^-40, far
// inside the 2^-9 spacing that the bf16 rounding of x^ must resolve.
__device__ __forceinline__ void rsqrt_pair(float ss_hi, float ss_lo, int D, float eps, float& y_hi, float& y_lo) {
  const float fd = static_cast<float>(D);
  const float q_hi = __fdiv_rn(ss_hi, fd);
  const float rem = __fmaf_rn(-q_hi, fd, ss_hi);  // exact: ss_hi - q_hi * D
  const float q_lo = __fdiv_rn(__fadd_rn(rem, ss_lo), fd);
  float s_hi, e;
  two_sum(q_hi, eps, s_hi, e);
  const float s_lo = __fadd_rn(e, q_lo);
  const float y0 = rsqrtf(s_hi);
  const float p = __fmul_rn(y0, y0);
  const float pe = __fmaf_rn(y0, y0, -p);  // y0^2 = p + pe exactly
  const float u = __fmaf_rn(s_hi, p, -1.f);
  const float t = __fadd_rn(u, __fmaf_rn(s_hi, pe, __fmul_rn(s_lo, p)));  // s y0^2 - 1
  const float corr = __fmul_rn(__fmul_rn(-0.5f, y0), t);
  two_sum(y0, corr, y_hi, y_lo);
}

// One CTA per row: x^ = x / sqrt(mean(x^2) + eps) * g rounded once to bf16.
// Because x is bf16, each x*x is exact in fp32 and the sum of squares is
// carried as an exact (hi, lo) pair; the scale is formed as a float pair and
// the final product is evaluated error-free (FMA) so that the bf16 rounding
// is the correctly rounded value of the real x^.  D % 8 == 0.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const __nv_bfloat16* __restrict__ gain,
                                                               __nv_bfloat16* __restrict__ out, int D, float eps,
                                                               int32_t* __restrict__ zero, int zero_count) {
  __shared__ float red_hi[kNormThreads / 32], red_lo[kNormThreads / 32];
  // Programmatic dependent launch: x may come from the preceding kernel.  The
  // projection kernel is released only once this row (and the gain) sit in
  // registers, so that its weight stream does not queue ahead of these loads.
  griddep_wait();
  if (blockIdx.x == 0)  // the projection's stream-K arrival counters start at zero
    for (int i = threadIdx.x; i < zero_count; i += kNormThreads) zero[i] = 0;
  const size_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * D);
  const uint4* gr = reinterpret_cast<const uint4*>(gain);
  uint4* orow = reinterpret_cast<uint4*>(out + row * D);
  const int nvec = D / 8;
  const bool in_regs = nvec <= kNormVecs * kNormThreads;
  uint4 xv[kNormVecs], gv4[kNormVecs];
#pragma unroll
  for (int j = 0; j < kNormVecs; ++j) {
    const int v = threadIdx.x + j * kNormThreads;
    const bool live = in_regs && v < nvec;
    xv[j] = live ? __ldg(xr + v) : make_uint4(0, 0, 0, 0);
    gv4[j] = live ? __ldg(gr + v) : make_uint4(0, 0, 0, 0);
  }
  float hi = 0.f, lo = 0.f;
  auto accumulate = [&](const uint4& u) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p[i]);
      float e;
      two_sum(hi, __fmul_rn(f.x, f.x), hi, e);
      lo = __fadd_rn(lo, e);
      two_sum(hi, __fmul_rn(f.y, f.y), hi, e);
      lo = __fadd_rn(lo, e);
    }
  };
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < kNormVecs; ++j) accumulate(xv[j]);
  } else {
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) accumulate(__ldg(xr + v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, o), ol = __shfl_xor_sync(0xffffffffu, lo, o);
    float e;
    two_sum(hi, oh, hi, e);
    lo = __fadd_rn(lo, __fadd_rn(e, ol));
  }
  if ((threadIdx.x & 31) == 0) {
    red_hi[threadIdx.x >> 5] = hi;
    red_lo[threadIdx.x >> 5] = lo;
  }
  __syncthreads();
  griddep_launch_dependents();
  // every thread forms the same scale from the per-warp pairs (fixed order)
  hi = red_hi[0];
  lo = red_lo[0];
#pragma unroll
  for (int w = 1; w < kNormThreads / 32; ++w) {
    float e;
    two_sum(hi, red_hi[w], hi, e);
    lo = __fadd_rn(lo, __fadd_rn(e, red_lo[w]));
  }
  float ss_hi, ss_lo;
  two_sum(hi, lo, ss_hi, ss_lo);
  float inv_hi, inv_lo;
  rsqrt_pair(ss_hi, ss_lo, D, eps, inv_hi, inv_lo);
  auto normalise = [&](const uint4& u, const uint4& gu) {
    const __nv_bfloat16* xp = reinterpret_cast<const __nv_bfloat16*>(&u);
    const __nv_bfloat16* gp = reinterpret_cast<const __nv_bfloat16*>(&gu);
    uint4 r;
    uint16_t* rp = reinterpret_cast<uint16_t*>(&r);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float xf = __bfloat162float(xp[i]), gv = __bfloat162float(gp[i]);
      // c = inv * g as an unevaluated pair, then x * c with its exact error
      const float c_hi = __fmul_rn(inv_hi, gv);
      const float c_lo = __fadd_rn(__fmaf_rn(inv_hi, gv, -c_hi), __fmul_rn(inv_lo, gv));
      const float p = __fmul_rn(xf, c_hi);
      const float e = __fadd_rn(__fmaf_rn(xf, c_hi, -p), __fmul_rn(xf, c_lo));
      rp[i] = bf16_round_pair(p, e);
    }
    return r;
  };
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < kNormVecs; ++j) {
      const int v = threadIdx.x + j * kNormThreads;
      if (v < nvec) orow[v] = normalise(xv[j], gv4[j]);
    }
  } else {
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) orow[v] = normalise(__ldg(xr + v), __ldg(gr + v));
  }
}

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

cudaError_t launch_rmsnorm(const void* x, const void* gain, void* out, int rows, int d_model, float eps,
                           int32_t* zero, int zero_count, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  // Same shared-memory carveout as the projection kernel that follows: an SM
  // cannot change its L1/shared split while a CTA of this kernel runs on it.
  cudaError_t e = cudaFuncSetAttribute(rmsnorm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, static_cast<const __nv_bfloat16*>(x),
                            static_cast<const __nv_bfloat16*>(gain), static_cast<__nv_bfloat16*>(out), d_model, eps,
                            zero, zero_count);
}

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
