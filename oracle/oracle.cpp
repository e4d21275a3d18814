// oracle.cpp — fp64 CPU oracle for one per-layer inner denoising step of
// block-wise (semi-autoregressive) diffusion-LLM decoding.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
// CPU-baseline leg of bench.py load this file's library.  The CUDA library never
// calls it and shares no code, header, table or constant with it.
//
// Every function is the plain definition from the pages, written out in fp64
// with no blocking or fusion:
//   * RMSNorm, the QKV projection and RoPE are the token-wise operators of
//     "LaCache: Exact Caching and Precision-Adaptive Inference for DLLMs",
//     §3.3.2, Eq. (1).
//   * Attention is the full bidirectional softmax attention that the naive
//     sampler recomputes at every step ("Fast-dLLM Block-wise DualCache",
//     section "Motivation"; LaCache Appendix B.2, Eq. (9)), written in two
//     passes (row max, then exp-sum).
//   * The online softmax state recurrence is LaCache §3.3.3, Eq. (2)-(6).
//   * The FACache build and reuse follow the definitions of LaCache §3.3.3
//     (each row's state over the keys of U, merged exactly with the fresh
//     keys); the tile-granular cache of its Algorithm 1 is restated as sets.
// Parallelism: OpenMP over independent outputs only; the arithmetic of each
// output is sequential in the order written.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// Round an fp64 value to the nearest bfloat16 value (ties to even), returned
// as fp64.  bfloat16 keeps the fp32 exponent range and 8 significant bits.
// The bf16 KV cache and the bf16 GEMM operand are the storage points where
// the step rounds.
double orc_bf16_round(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  const double ax = fabs(x);
  int e;
  frexp(ax, &e);  // ax = f * 2^e with f in [0.5, 1)
  // Spacing of bf16 values around ax: 8 significant bits for normal values
  // (exponent >= -125 in frexp terms), fixed spacing 2^-133 below that.
  int ulp_exp = e - 8;
  if (ulp_exp < -133) ulp_exp = -133;
  const double ulp = ldexp(1.0, ulp_exp);
  const double q = ax / ulp;  // exact: scaling by a power of two
  double r = floor(q);
  const double frac = q - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double y = r * ulp;
  // Largest finite bf16 is (2 - 2^-7) * 2^127; anything that rounds above it overflows.
  const double max_bf16 = ldexp(255.0, 120);
  if (y > max_bf16) y = INFINITY;
  return x < 0 ? -y : y;
}

void orc_bf16_round_array(double* a, int64_t n) {
  for (int64_t i = 0; i < n; ++i) a[i] = orc_bf16_round(a[i]);
}

// RMSNorm (LaCache §3.3.2, "attention norm"):
//   out[r][c] = x[r][c] / sqrt(mean_c(x[r][c]^2) + eps) * g[c]
void orc_rmsnorm(const double* x, int64_t rows, int64_t D, const double* g, double eps, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t c = 0; c < D; ++c) ss += x[r * D + c] * x[r * D + c];
    const double inv = 1.0 / sqrt(ss / (double)D + eps);
    for (int64_t c = 0; c < D; ++c) out[r * D + c] = x[r * D + c] * inv * g[c];
  }
}

// Linear projection without bias (LaCache Eq. (1), H^ W):
//   out[r][n] = sum_k x[r][k] * W[n][k]      (W stored [nout][D], row-major)
// Each output is the plain sum over k in order, starting from 0.  Eight
// outputs of a row are summed side by side (eight independent running sums,
// so the additions of different outputs overlap in the pipeline); the last
// group repeats the last weight row for the missing outputs and drops them.
void orc_linear(const double* x, int64_t rows, int64_t D, const double* W, int64_t nout, double* out) {
  const int64_t ngroups = (nout + 7) / 8;
#pragma omp parallel for schedule(static)
  for (int64_t gi = 0; gi < ngroups; ++gi) {
    const double* w[8];
    for (int i = 0; i < 8; ++i) {
      const int64_t n = gi * 8 + i < nout ? gi * 8 + i : nout - 1;
      w[i] = W + n * D;
    }
    for (int64_t r = 0; r < rows; ++r) {
      const double* xr = x + r * D;
      double acc[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
      for (int64_t k = 0; k < D; ++k)
        for (int i = 0; i < 8; ++i) acc[i] += xr[k] * w[i][k];
      for (int i = 0; i < 8 && gi * 8 + i < nout; ++i) out[r * nout + gi * 8 + i] = acc[i];
    }
  }
}

// Rotary position embedding (LaCache Eq. (1), RoPE), rotate-half pairing:
// for each head the pair (i, i + d/2), i < d/2, is rotated by the angle
// pos * theta^(-2i/d).  t is [rows][H][d], rotated in place.
void orc_rope(double* t, int64_t rows, int64_t H, int64_t d, const int64_t* pos, double theta) {
  const int64_t half = d / 2;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      double* v = t + (r * H + h) * d;
      for (int64_t i = 0; i < half; ++i) {
        const double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        const double ang = (double)pos[r] * inv_freq;
        const double c = cos(ang), s = sin(ang);
        const double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
      }
    }
  }
}

// Full bidirectional attention, two-pass softmax (no mask):
//   S[j] = scale * <q_r, k_j>,  m = max_j S[j],  l = sum_j exp(S[j] - m),
//   O_r = sum_j exp(S[j] - m) v_j / l,  L_r = m + ln l.
// q [nq][H][d]; k, v [nk][H][d]; O [nq][H][d]; L [nq][H] (nullable).
void orc_attention(const double* q, int64_t nq, const double* k, const double* v, int64_t nk, int64_t H, int64_t d,
                   double scale, double* O, double* L) {
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int64_t r = 0; r < nq; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      std::vector<double> S(nk);
      const double* qr = q + (r * H + h) * d;
      double m = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        const double* kj = k + (j * H + h) * d;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qr[c] * kj[c];
        S[j] = scale * dot;
        if (S[j] > m) m = S[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j < nk; ++j) l += exp(S[j] - m);
      double* o = O + (r * H + h) * d;
      for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        const double p = exp(S[j] - m) / l;
        const double* vj = v + (j * H + h) * d;
        for (int64_t c = 0; c < d; ++c) o[c] += p * vj[c];
      }
      if (L) L[r * H + h] = m + log(l);
    }
  }
}

// One online-softmax update (LaCache Eq. (2)-(6)) of the per-row state
// (m, l, Ot) with the keys listed in `keys` (a tile), for one (row, head).
static void online_update(const double* qr, const double* k, const double* v, int64_t H, int64_t h, int64_t d,
                          double scale, const int64_t* keys, int64_t nkeys, double* m, double* l, double* Ot) {
  if (nkeys == 0) return;
  std::vector<double> S(nkeys);
  double rm = -INFINITY;  // RM(S): row max of the tile
  for (int64_t t = 0; t < nkeys; ++t) {
    const double* kj = k + (keys[t] * H + h) * d;
    double dot = 0.0;
    for (int64_t c = 0; c < d; ++c) dot += qr[c] * kj[c];
    S[t] = scale * dot;
    if (S[t] > rm) rm = S[t];
  }
  const double m_new = (*m > rm) ? *m : rm;                      // Eq. (2)
  const double alpha = (*m == -INFINITY) ? 0.0 : exp(*m - m_new);  // Eq. (3); empty state has weight 0
  double rs = 0.0;
  for (int64_t c = 0; c < d; ++c) Ot[c] *= alpha;  // first term of Eq. (6)
  for (int64_t t = 0; t < nkeys; ++t) {
    const double p = exp(S[t] - m_new);  // Eq. (4)
    rs += p;                             // RS(P~)
    const double* vj = v + (keys[t] * H + h) * d;
    for (int64_t c = 0; c < d; ++c) Ot[c] += p * vj[c];  // second term of Eq. (6)
  }
  *l = alpha * (*l) + rs;  // Eq. (5)
  *m = m_new;
}

// Online-softmax attention over all keys (LaCache Eq. (2)-(6)) with keys
// visited in tiles of `bc` following the permutation `order` of tile indices
// (nullable: natural order).  O = diag(l)^-1 Ot, L = m + ln l.
void orc_attention_online(const double* q, int64_t nq, const double* k, const double* v, int64_t nk, int64_t H,
                          int64_t d, double scale, int64_t bc, const int64_t* order, double* O, double* L) {
  const int64_t ntiles = (nk + bc - 1) / bc;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int64_t r = 0; r < nq; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      double m = -INFINITY, l = 0.0;
      std::vector<double> Ot(d, 0.0);
      std::vector<int64_t> keys;
      for (int64_t ti = 0; ti < ntiles; ++ti) {
        const int64_t t = order ? order[ti] : ti;
        keys.clear();
        for (int64_t j = t * bc; j < nk && j < (t + 1) * bc; ++j) keys.push_back(j);
        online_update(q + (r * H + h) * d, k, v, H, h, d, scale, keys.data(), (int64_t)keys.size(), &m, &l,
                      Ot.data());
      }
      for (int64_t c = 0; c < d; ++c) O[(r * H + h) * d + c] = Ot[c] / l;
      if (L) L[r * H + h] = m + log(l);
    }
  }
}

// FACache build (LaCache §3.3.3; Algorithm 1 with GenStep = True), token
// granular: for each query row listed in `rows` and each head, the online
// state (m, l, Ot) after streaming, in tiles of `bc` keys, every key of the
// sequence that lies outside the current block [c_lo, c_hi).  The reference
// max is the maximum over those keys only.  q [nrows][H][d] holds the rows'
// queries; k, v [nk][H][d] hold all keys of the sequence.
// Outputs: m, l [nrows][H]; Ot [nrows][H][d].
void orc_state_build(const double* q, int64_t nrows, const double* k, const double* v, int64_t nk, int64_t H,
                     int64_t d, double scale, int64_t c_lo, int64_t c_hi, int64_t bc, double* m_out, double* l_out,
                     double* Ot_out) {
  const int64_t ntiles = (nk + bc - 1) / bc;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      double m = -INFINITY, l = 0.0;
      double* Ot = Ot_out + (r * H + h) * d;
      for (int64_t c = 0; c < d; ++c) Ot[c] = 0.0;
      std::vector<int64_t> keys;
      for (int64_t t = 0; t < ntiles; ++t) {
        keys.clear();
        for (int64_t j = t * bc; j < nk && j < (t + 1) * bc; ++j)
          if (j < c_lo || j >= c_hi) keys.push_back(j);  // keys of the invariant set only
        online_update(q + (r * H + h) * d, k, v, H, h, d, scale, keys.data(), (int64_t)keys.size(), &m, &l, Ot);
      }
      m_out[r * H + h] = m;
      l_out[r * H + h] = l;
    }
  }
}

// FACache reuse (LaCache §3.3.3; Algorithm 1 with GenStep = False), token
// granular: each listed row starts from its cached state (m, l, Ot) and
// streams only the keys of the current block [c_lo, c_hi), in tiles of `bc`;
// then O = diag(l)^-1 Ot and L = m + ln l.  Inputs as for orc_state_build.
void orc_state_merge(const double* q, int64_t nrows, const double* k, const double* v, int64_t nk, int64_t H,
                     int64_t d, double scale, int64_t c_lo, int64_t c_hi, int64_t bc, const double* m_in,
                     const double* l_in, const double* Ot_in, double* O, double* L) {
  (void)nk;
#pragma omp parallel for collapse(2) schedule(dynamic, 4)
  for (int64_t r = 0; r < nrows; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      double m = m_in[r * H + h], l = l_in[r * H + h];
      std::vector<double> Ot(Ot_in + (r * H + h) * d, Ot_in + (r * H + h + 1) * d);
      std::vector<int64_t> keys;
      for (int64_t t0 = c_lo; t0 < c_hi; t0 += bc) {
        keys.clear();
        for (int64_t j = t0; j < c_hi && j < t0 + bc; ++j) keys.push_back(j);
        online_update(q + (r * H + h) * d, k, v, H, h, d, scale, keys.data(), (int64_t)keys.size(), &m, &l,
                      Ot.data());
      }
      for (int64_t c = 0; c < d; ++c) O[(r * H + h) * d + c] = Ot[c] / l;
      if (L) L[r * H + h] = m + log(l);
    }
  }
}

// The FACache of LaCache §3.3.3 at tile granularity, for one sequence of N
// tokens whose current block is C = [c_lo, c_hi).  Rows are grouped in tiles
// of br and keys in tiles of bc; a tile that holds any token of C is fresh as
// a whole.  Written as sets: R_f / K_f = the rows / keys of fresh tiles, and
// K_u = every other key.
//   genstep != 0 (building the cache): every row's output is its attention
//     over all N keys; every row outside R_f also stores, in (mc, lc, Oc), its
//     online-softmax state over K_u.
//   genstep == 0 (reusing it): a row outside R_f outputs the exact merge of its
//     stored state with its state over K_f; a row of R_f attends over all keys.
// Every row produces O and L.  q, k, v [N][H][d]; mc, lc [N][H], Oc [N][H][d].
void orc_alg1(const double* q, const double* k, const double* v, int64_t N, int64_t H, int64_t d, double scale,
              int64_t c_lo, int64_t c_hi, int64_t br, int64_t bc, int genstep, double* mc, double* lc, double* Oc,
              double* O, double* L) {
  // the tile-granular sets
  std::vector<char> row_fresh(N, 0);
  std::vector<int64_t> keys_all, keys_fresh, keys_kept;
  auto tile_holds_block = [&](int64_t t, int64_t size) {
    const int64_t lo = t * size, hi = (lo + size < N) ? lo + size : N;
    return lo < c_hi && c_lo < hi;
  };
  for (int64_t r = 0; r < N; ++r) row_fresh[r] = tile_holds_block(r / br, br) ? 1 : 0;
  for (int64_t j = 0; j < N; ++j) {
    keys_all.push_back(j);
    (tile_holds_block(j / bc, bc) ? keys_fresh : keys_kept).push_back(j);
  }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t r = 0; r < N; ++r) {
    for (int64_t h = 0; h < H; ++h) {
      const double* qr = q + (r * H + h) * d;
      const int64_t rh = r * H + h;
      double m = -INFINITY, l = 0.0;
      std::vector<double> Ot(d, 0.0);
      if (genstep || row_fresh[r]) {  // attention over every key
        online_update(qr, k, v, H, h, d, scale, keys_all.data(), (int64_t)keys_all.size(), &m, &l, Ot.data());
      } else {  // the stored state, merged with the fresh keys
        m = mc[rh];
        l = lc[rh];
        for (int64_t c = 0; c < d; ++c) Ot[c] = Oc[rh * d + c];
        online_update(qr, k, v, H, h, d, scale, keys_fresh.data(), (int64_t)keys_fresh.size(), &m, &l, Ot.data());
      }
      for (int64_t c = 0; c < d; ++c) O[rh * d + c] = Ot[c] / l;
      L[rh] = m + log(l);
      if (genstep && !row_fresh[r]) {  // store the state over the kept keys
        double cm = -INFINITY, cl = 0.0;
        std::vector<double> cO(d, 0.0);
        online_update(qr, k, v, H, h, d, scale, keys_kept.data(), (int64_t)keys_kept.size(), &cm, &cl, cO.data());
        mc[rh] = cm;
        lc[rh] = cl;
        for (int64_t c = 0; c < d; ++c) Oc[rh * d + c] = cO[c];
      }
    }
  }
}

// The softmax over a row of logits, summarised (LaCache §3.4, the sampling stage; the
// quantities a confidence sampler reads): lse = m + log sum_v exp(z_v - m) with m the row
// max, argmax = the lowest v with z_v = m, p_max = exp(m - lse).  Two passes, fp64.
void orc_softmax_stats(const double* z, int64_t rows, int64_t V, double* lse, int64_t* argmax, double* pmax) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* zr = z + r * V;
    double m = zr[0];
    int64_t am = 0;
    for (int64_t v = 1; v < V; ++v)
      if (zr[v] > m) {
        m = zr[v];
        am = v;
      }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += exp(zr[v] - m);
    lse[r] = m + log(s);
    argmax[r] = am;
    pmax[r] = exp(m - lse[r]);
  }
}

// ---- FP8 (e4m3) for the FFN's per-group quantisation (LaCache §3.4, Eq. (7)-(8)).
// e4m3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 holds the
// subnormals m/8 * 2^-6; the largest finite magnitude is 1.75 * 2^8 = 448; no infinities.

// The value of an e4m3 code (the two NaN codes give NaN).
double orc_e4m3_decode(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

// Round to the nearest e4m3 value, ties to the even mantissa, magnitudes beyond 448
// saturated to 448 (the clip of Eq. (7) with Q_max = 448).
double orc_e4m3_round(double x) {
  const double a = fabs(x);
  if (a == 0.0) return x;
  int e;
  frexp(a, &e);       // a = f * 2^e, f in [0.5, 1)
  int ex = e - 1;     // a in [2^ex, 2^(ex+1))
  if (ex < -6) ex = -6;  // the subnormal spacing below 2^-6
  const double step = ldexp(1.0, ex - 3);
  double r = nearbyint(a / step) * step;  // the default rounding mode: to nearest even
  if (r > 448.0) r = 448.0;
  return x < 0 ? -r : r;
}

// Eq. (7)-(8) for rows of x [rows][cols] in groups of `group` columns: scale_g =
// max_g |x| / 448 and q = e4m3(x / scale_g), each decision taken in fp32 (x rounded to
// fp32 first, the division correctly rounded), as the kernels take it.  Writes the
// dequantised values q * scale_g and the scales [rows][cols / group].
void orc_quant_groups(const double* x, int64_t rows, int64_t cols, int64_t group, double* deq, double* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t g0 = 0; g0 < cols; g0 += group) {
      float amax = 0.f;
      for (int64_t c = g0; c < g0 + group; ++c) amax = fmaxf(amax, fabsf((float)x[r * cols + c]));
      const float sc = amax / 448.f;
      scales[r * (cols / group) + g0 / group] = sc;
      for (int64_t c = g0; c < g0 + group; ++c) {
        const float t = sc > 0.f ? (float)x[r * cols + c] / sc : 0.f;
        deq[r * cols + c] = orc_e4m3_round((double)t) * (double)sc;
      }
    }
  }
}

// The input of the AddNorm's quantisation, in the precision the quantisation decides in:
// x2 = RMSNorm(h) g taken as the kernels take it in fp32, with 1 / rms correctly rounded to
// fp32 (from the exact fp64 mean) and the two products rounded to fp32 in the order (h *
// inv) * g.  Returns the fp32 values as doubles.
void orc_rmsnorm_f32(const double* h, int64_t rows, int64_t D, const double* g, double eps, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t c = 0; c < D; ++c) ss += h[r * D + c] * h[r * D + c];
    const double ms = ss / (double)D;  // the mean square
    const float inv = (float)(1.0 / sqrt(ms + eps));
    for (int64_t c = 0; c < D; ++c) {
      const float t = (float)h[r * D + c] * inv;
      out[r * D + c] = (double)(t * (float)g[c]);
    }
  }
}

// Dequantise e4m3 codes [rows][cols] with one scale per block of br x bc: [rows / br][cols / bc].
void orc_dequant_blocks(const uint8_t* codes, int64_t rows, int64_t cols, int64_t br, int64_t bc,
                        const float* scales, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = orc_e4m3_decode(codes[r * cols + c]) * (double)scales[(r / br) * (cols / bc) + c / bc];
}

}  // extern "C"
