/*
 * oracle.cpp -- plain, slow, double-precision CPU oracle for the draft-block
 * select-and-verify step of DFlash 2 block drafting.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library never
 * links, includes or calls it; the two share no header, helper, table or
 * constant. Its inputs are the caller's raw bf16 (uint16 bit patterns) or
 * fp32 bytes; every element is widened to double (exact) before any
 * arithmetic, and every result is computed in double.
 *
 * Sources, cited by page title and section / equation / table:
 *   [Blog]   "DFlash 2: Keep Drafting Parallel" (Chinese translation of the
 *            Inco AI blog, "DFlash 2：保持并行草案生成")
 *   [ZhTW]   "DFlash 2 讓 Qwen3.8-27B 快了兩倍：同模型、同輸出、同一張卡，純粹靠更聰明的推理"
 *   [Digest] "给 Qwen3.8-27B 配个"草稿加速器"：DFlash2 并行投机解码解读"
 *
 * What pins each function (tests/test_oracle_*.py):
 *   orc_logits, orc_topk ..... numpy float64 matmul and lexsort on the same bytes
 *   orc_gate ................. closed-form special cases (zero weights, one-hot
 *                              weights, sign flip); the sigmoid form itself is a
 *                              reading (the pages name a "context gate" only)
 *   orc_pair_scores .......... one-hot closed forms, linearity, A = 0 gives U
 *   orc_path_viterbi ......... brute force over all K^(L-1) paths
 *   orc_path_greedy .......... hand-worked golden lattice; A = 0 gives top-1
 *   orc_path_sample_joint .... brute force over all K^P paths: the product of the drawn
 *                              conditionals is the path's exact probability; chi-square of
 *                              drawn paths; T -> 0 gives the Viterbi path
 *   orc_verify_greedy ........ equality with target-argmax decoding
 *   orc_verify_sampling ...... chi-square of emitted-token marginals against
 *                              the target softmax (1e6 draws; and redraws over a
 *                              vocabulary of 9192 tokens); limiting cases
 *   orc_redraw_uniforms ...... enumeration: on a grid of n uniforms each token is
 *                              drawn n * (its residual probability) times, within one
 *   orc_philox4x64 ........... numpy.random.Philox raw output
 *   accept length ............ closed form that reproduces the [Blog] Table 1
 *                              verify lengths 4.27 / 6.79
 *   orc_conv2tap ............. identity and shift kernels (zero correction), one
 *                              correction group at a time, the correction read from
 *                              the position's own row, and the [Blog]'s parameter count
 *
 * Tie rule everywhere: among equal values the lower token id wins.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum { ORC_BF16 = 0, ORC_FP32 = 1 };

const double kInf = std::numeric_limits<double>::infinity();

/* Exact widening of one stored element to double. */
inline double widen(const void* p, int dtype, int64_t i) {
  if (dtype == ORC_BF16) {
    uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16;
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return static_cast<double>(f);
  }
  return static_cast<double>(static_cast<const float*>(p)[i]);
}

/* (value desc, id asc): true when candidate (va, ia) ranks before (vb, ib). */
inline bool ranks_before(double va, int64_t ia, double vb, int64_t ib) {
  return va > vb || (va == vb && ia < ib);
}

inline double rel(double margin, double value) {
  return margin / std::max(1.0, std::fabs(value));
}

/* ---- Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3", SC'11). Ten rounds of the 4x64 Philox S-box keyed by
 * a Weyl sequence. Written from the published definition. */
const uint64_t kPhiloxM0 = 0xD2E7470EE14C6C93ULL;
const uint64_t kPhiloxM1 = 0xCA5A826395121157ULL;
const uint64_t kPhiloxW0 = 0x9E3779B97F4A7C15ULL;
const uint64_t kPhiloxW1 = 0xBB67AE8584CAA73BULL;

void philox4x64_10(const uint64_t in[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t c0 = in[0], c1 = in[1], c2 = in[2], c3 = in[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    unsigned __int128 p0 = static_cast<unsigned __int128>(kPhiloxM0) * c0;
    unsigned __int128 p1 = static_cast<unsigned __int128>(kPhiloxM1) * c2;
    uint64_t hi0 = static_cast<uint64_t>(p0 >> 64), lo0 = static_cast<uint64_t>(p0);
    uint64_t hi1 = static_cast<uint64_t>(p1 >> 64), lo1 = static_cast<uint64_t>(p1);
    uint64_t n0 = hi1 ^ c1 ^ k0;
    uint64_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform in (0,1) from the top 23 bits of a 64-bit word: (2j+1) * 2^-24 with
 * j < 2^23, an odd 24-bit integer times a power of two, so exact in fp32 and fp64. */
inline double u01(uint64_t x) {
  return (static_cast<double>(x >> 41) + 0.5) * (1.0 / 8388608.0);
}

/* Counter layout shared by definition (not by code) with the GPU path:
 *   key     = (seed, 0)
 *   accept  : counter (0, t, b, 0), word 0           -- position t = 1..L-1
 *   redraw  : counter (0, t, b, 1), word 0           -- the redraw's one uniform
 *   path    : counter (0, t, b, 3), word 0           -- the sampled path's draw at t
 * The redraw from row t-1 uses position t; the bonus row L-1 uses t = L. */
double uniform_counter(uint64_t seed, int64_t b, int t, uint64_t idx, uint64_t stream, int word) {
  uint64_t ctr[4] = {idx, static_cast<uint64_t>(t), static_cast<uint64_t>(b), stream};
  uint64_t key[2] = {seed, 0ULL};
  uint64_t o[4];
  philox4x64_10(ctr, key, o);
  return u01(o[word]);
}

double uniform_accept(uint64_t seed, int64_t b, int t) { return uniform_counter(seed, b, t, 0, 0, 0); }

double uniform_redraw(uint64_t seed, int64_t b, int t) { return uniform_counter(seed, b, t, 0, 1, 0); }

double uniform_path(uint64_t seed, int64_t b, int t) { return uniform_counter(seed, b, t, 0, 3, 0); }

/* log-sum-exp of z/T over one row, in double. */
double row_lse(const void* Z, int zdtype, int64_t off, int64_t V, double T) {
  double m = -kInf;
  for (int64_t v = 0; v < V; ++v) m = std::max(m, widen(Z, zdtype, off + v) / T);
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) s += std::exp(widen(Z, zdtype, off + v) / T - m);
  return m + std::log(s);
}

/* Inverse-CDF draw over the weights w[0..n) (w >= 0) with one uniform u: the first index
 * whose cumulative weight exceeds u * sum(w) (in index order); if rounding leaves none, the
 * last index with weight. Returns -1 when every weight is zero. margin = the distance of
 * the target u * sum(w) to the nearest cumulative boundary, relative to the sum. */
int64_t inverse_cdf(const std::vector<double>& w, double u, double* margin) {
  double total = 0.0;
  int64_t last = -1;
  for (size_t i = 0; i < w.size(); ++i) {
    total += w[i];
    if (w[i] > 0.0) last = static_cast<int64_t>(i);
  }
  *margin = kInf;
  if (last < 0) return -1;
  const double target = u * total;
  double cum = 0.0;
  int64_t pick = -1;
  for (size_t i = 0; i < w.size(); ++i) {
    if (!(w[i] > 0.0)) continue;
    cum += w[i];
    *margin = std::min(*margin, std::fabs(cum - target) / total);
    if (pick < 0 && cum > target) pick = static_cast<int64_t>(i);
  }
  return pick < 0 ? last : pick;
}

/* An exact draw from p = softmax(z/T) over one row with token excl removed (excl < 0:
 * none) and renormalised: the weights exp(z_v/T - max) of every other token, cumulated in
 * vocabulary order, against the one uniform u (inverse_cdf). margin as inverse_cdf's. */
int64_t redraw(const void* Z, int zdtype, int64_t off, int64_t V, double T, double u, int64_t excl,
               double* margin) {
  double m = -kInf;
  for (int64_t v = 0; v < V; ++v) m = std::max(m, widen(Z, zdtype, off + v) / T);
  std::vector<double> w(V);
  for (int64_t v = 0; v < V; ++v) w[v] = (v != excl) ? std::exp(widen(Z, zdtype, off + v) / T - m) : 0.0;
  const int64_t y = inverse_cdf(w, u, margin);
  return y < 0 ? 0 : y;
}

/* An exact draw from the residual r(v) = max(0, p(v) - q(v)) renormalised, with
 * p = softmax(z/T) over the row and q a proposal that is nonzero only on the K listed
 * candidates (cand[k] with probability qv[k]); K = 0 draws from p itself. The weights r(v),
 * cumulated in vocabulary order, against the one uniform u (inverse_cdf). For a proposal
 * that puts all its mass on one token this is redraw() with that token excluded (the
 * weights differ from redraw()'s by the row's constant normaliser). */
int64_t redraw_residual(const void* Z, int zdtype, int64_t off, int64_t V, double T, double u,
                        const int32_t* cand, const double* qv, int K, double* margin) {
  const double lse = row_lse(Z, zdtype, off, V, T);
  std::vector<double> w(V);
  for (int64_t v = 0; v < V; ++v) w[v] = std::exp(widen(Z, zdtype, off + v) / T - lse);
  for (int k = 0; k < K; ++k)
    if (cand[k] >= 0 && cand[k] < V) w[cand[k]] = std::max(0.0, w[cand[k]] - qv[k]);
  const int64_t y = inverse_cdf(w, u, margin);
  return y < 0 ? 0 : y;
}

/* ---- E4M3, the OCP 8-bit floating-point format ("OCP 8-bit Floating Point
 * Specification (OFP8)", 2023): 1 sign, 4 exponent (bias 7) and 3 mantissa bits; normals
 * (8 + m) 2^(e - 10) for e = 1..15 up to 448 = 1.75 * 2^8, subnormals m 2^-9, no
 * infinities, S.1111.111 is NaN. */
double e4m3_value(uint8_t b) {
  const int sgn = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const double v = (e == 0) ? std::ldexp(static_cast<double>(m), -9)
                            : std::ldexp(static_cast<double>(8 + m), e - 10);
  return sgn ? -v : v;
}

/* x (|x| <= 448) rounded to E4M3, to nearest with ties to even: the grid spacing is
 * 2^(E - 3) in the binade [2^E, 2^(E+1)) for E >= -6 and 2^-9 below. */
uint8_t e4m3_round(double x) {
  const uint8_t sgn = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  int E = -6;
  if (a >= std::ldexp(1.0, -6)) {
    int ex;
    std::frexp(a, &ex);  // a = f 2^ex, f in [0.5, 1)
    E = ex - 1;
  }
  const double q = std::ldexp(1.0, E - 3);
  const double v = std::nearbyint(a / q) * q;  // a / q is exact (a power of two)
  if (v == 0.0) return sgn;
  if (v < std::ldexp(1.0, -6))
    return static_cast<uint8_t>(sgn | static_cast<int>(v / std::ldexp(1.0, -9)));
  int ex;
  std::frexp(v, &ex);
  const int e = ex - 1 + 7;                                             // biased exponent
  const int m = static_cast<int>(v / std::ldexp(1.0, ex - 1 - 3)) - 8;  // 3 mantissa bits
  return static_cast<uint8_t>(sgn | (e << 3) | m);
}

/* The power-of-two scale of a row quantised to E4M3: the smallest 2^e with
 * amax <= 448 * 2^e (448 is E4M3's largest value); 1 when amax is 0 or below 2^-100. */
double e4m3_row_scale(double amax) {
  if (!(amax >= std::ldexp(1.0, -100))) return 1.0;
  int E;
  const double f = std::frexp(amax, &E);  // amax = f 2^E, f in [0.5, 1); 448 = 0.875 2^9
  return std::ldexp(1.0, E - 9 + (f > 0.875 ? 1 : 0));
}

}  // namespace

extern "C" {

int orc_abi_version() { return 1; }

/* E4M3 bytes to double, and doubles (|x| <= 448) to E4M3 bytes, for the format pins. */
void orc_e4m3_decode(const uint8_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(b[i]);
}
void orc_e4m3_encode(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round(x[i]);
}

/* Rows of the hidden states quantised for the E4M3 LM head: per row a power-of-two
 * scale s (e4m3_row_scale of the row's largest magnitude) and q[k] = E4M3(h[k] / s).
 * h [*, d] of dtype; rows [n]; q [n][d] bytes; scale [n]. */
int orc_quantize_rows_e4m3(int dtype, const void* h, int64_t d, const int64_t* rows, int64_t n,
                           uint8_t* q, double* scale) {
  if (d <= 0 || n < 0 || (dtype != ORC_BF16 && dtype != ORC_FP32)) return -1;
  for (int64_t i = 0; i < n; ++i) {
    double amax = 0.0;
    for (int64_t k = 0; k < d; ++k)
      amax = std::max(amax, std::fabs(widen(h, dtype, rows[i] * d + k)));
    const double s = e4m3_row_scale(amax);
    scale[i] = s;
    for (int64_t k = 0; k < d; ++k) q[i * d + k] = e4m3_round(widen(h, dtype, rows[i] * d + k) / s);
  }
  return 0;
}

/* Draft logits of the E4M3 LM head: W stored [V][d] as E4M3 bytes with one scale per
 * vocabulary entry, the rows quantised as above:
 * u[i][v] = s_h[i] s_w[v] sum_k E4M3(q[i][k]) E4M3(Wq[v][k]), in double. */
int orc_logits_e4m3(const uint8_t* q, const double* h_scale, const uint8_t* Wq,
                    const float* w_scale, int64_t d, int64_t V, int64_t n, double* u,
                    int nthreads) {
  if (d <= 0 || V <= 0 || n < 0) return -1;
  std::vector<double> hd(static_cast<size_t>(n) * d);
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = 0; k < d; ++k) hd[i * d + k] = e4m3_value(q[i * d + k]);
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    std::vector<double> w(d);
#pragma omp for schedule(dynamic, 64)
    for (int64_t v = 0; v < V; ++v) {
      for (int64_t k = 0; k < d; ++k) w[k] = e4m3_value(Wq[v * d + k]);
      for (int64_t i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k) acc += hd[i * d + k] * w[k];
        u[i * V + v] = acc * h_scale[i] * static_cast<double>(w_scale[v]);
      }
    }
  }
  return 0;
}

/* Draft logits, [Blog] §"A lightweight path selector": U_t(b) is the drafter's
 * own logit for b, i.e. the shared LM head applied to the position's hidden
 * state. u[i][v] = sum_{k<d} h[rows[i]][k] * W[k][v], W stored [d][V].
 * Each output is one dot product accumulated in k order; the vocabulary is
 * split across threads only to use the cores. */
int orc_logits(int dtype, const void* h, const void* W, int64_t d, int64_t V,
               const int64_t* rows, int64_t n, double* u, int nthreads) {
  if (d <= 0 || V <= 0 || n < 0 || (dtype != ORC_BF16 && dtype != ORC_FP32)) return -1;
  std::vector<double> hd(static_cast<size_t>(n) * d);
  for (int64_t i = 0; i < n; ++i)
    for (int64_t k = 0; k < d; ++k) hd[i * d + k] = widen(h, dtype, rows[i] * d + k);
  const int64_t CH = 512;
  const int64_t nch = (V + CH - 1) / CH;
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    std::vector<double> wrow(CH);
    std::vector<double> acc(static_cast<size_t>(n) * CH);
#pragma omp for schedule(dynamic, 1)
    for (int64_t c = 0; c < nch; ++c) {
      const int64_t v0 = c * CH;
      const int64_t w = std::min(CH, V - v0);
      std::fill(acc.begin(), acc.end(), 0.0);
      for (int64_t k = 0; k < d; ++k) {
        for (int64_t j = 0; j < w; ++j) wrow[j] = widen(W, dtype, k * V + v0 + j);
        for (int64_t i = 0; i < n; ++i) {
          const double hk = hd[i * d + k];
          double* a = acc.data() + i * CH;
          for (int64_t j = 0; j < w; ++j) a[j] += hk * wrow[j];
        }
      }
      for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < w; ++j) u[i * V + v0 + j] = acc[i * CH + j];
    }
  }
  return 0;
}

/* Keep top-K, [Blog] §"The right tokens are already there" and §"A lightweight
 * path selector" (K = 16): the K largest logits of a row, ordered by
 * (value desc, id asc). gap[i] = u_K - u_{K+1} (the boundary margin; +inf when
 * V == K). */
int orc_topk(const double* u, int64_t n, int64_t V, int K, int32_t* ids, double* U, double* gap) {
  if (K <= 0 || V < K) return -1;
  std::vector<int64_t> idx(V);
  const int64_t keep = std::min<int64_t>(V, K + 1);
  for (int64_t i = 0; i < n; ++i) {
    const double* row = u + i * V;
    for (int64_t v = 0; v < V; ++v) idx[v] = v;
    std::partial_sort(idx.begin(), idx.begin() + keep, idx.end(), [row](int64_t a, int64_t b) {
      return ranks_before(row[a], a, row[b], b);
    });
    for (int k = 0; k < K; ++k) {
      ids[i * K + k] = static_cast<int32_t>(idx[k]);
      U[i * K + k] = row[idx[k]];
    }
    gap[i] = (V > K) ? row[idx[K - 1]] - row[idx[K]] : kInf;
  }
  return 0;
}

/* Context gate H(h_t), [Blog] §"A lightweight path selector": the pages name a
 * gate computed from the position's hidden state that decides which of the
 * rank dimensions count; its form is not printed. Reading taken:
 * g[i][j] = sigmoid(sum_k Wg[j][k] * h[rows[i]][k]), Wg stored [r][d]. */
int orc_gate(int dtype, const void* h, const void* Wg, int64_t d, int64_t r,
             const int64_t* rows, int64_t n, double* g) {
  if (d <= 0 || r <= 0 || n < 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    for (int64_t j = 0; j < r; ++j) {
      double x = 0.0;
      for (int64_t k = 0; k < d; ++k) x += widen(Wg, dtype, j * d + k) * widen(h, dtype, rows[i] * d + k);
      g[i * r + j] = 1.0 / (1.0 + std::exp(-x));
    }
  }
  return 0;
}

/* Bilinear pair scores, [Blog] §"A lightweight path selector", eq.
 * S_t(a,b) = U_t(b) + < A(a) (.) H(h_t), B(b) >, and [ZhTW] §2 (same eq.).
 * P = L-1 draft positions, position t = p+1. The predecessor of position 1 is
 * the last verified token x0 ("start from the last verified token"), so every
 * a-row of p = 0 holds S_1(x0, .). For p >= 1 the predecessor a ranges over
 * the candidates of position p. Output S[p][a][b]. */
int orc_pair_scores(int dtype, const void* A, const void* Bt, int64_t r, int P, int K,
                    const int32_t* ids, const double* U, const double* g, int32_t x0, double* S) {
  if (r <= 0 || P < 1 || K < 1) return -1;
  for (int p = 0; p < P; ++p) {
    for (int a = 0; a < K; ++a) {
      const int64_t tok_a = (p == 0) ? x0 : ids[(p - 1) * K + a];
      for (int bb = 0; bb < K; ++bb) {
        const int64_t tok_b = ids[p * K + bb];
        double s = 0.0;
        for (int64_t j = 0; j < r; ++j)
          s += widen(A, dtype, tok_a * r + j) * g[p * r + j] * widen(Bt, dtype, tok_b * r + j);
        S[(static_cast<int64_t>(p) * K + a) * K + bb] = U[p * K + bb] + s;
      }
    }
  }
  return 0;
}

/* Greedy traversal, [Blog] §"A lightweight path selector": from the last
 * verified token, follow the best successor at each step.
 * x_1 = argmax_b S_1(x0,b); x_t = argmax_b S_t(x_{t-1}, b).
 * score = sum of the chosen S values (left to right). margin = smallest
 * relative gap best-vs-second among the decisions taken. */
int orc_path_greedy(int P, int K, const double* S, const int32_t* ids, int32_t* path,
                    int32_t* path_idx, double* score, double* margin) {
  if (P < 1 || K < 1) return -1;
  int a = 0;
  double total = 0.0, mm = kInf;
  for (int p = 0; p < P; ++p) {
    const double* row = S + (static_cast<int64_t>(p) * K + a) * K;
    int best = 0;
    for (int b = 1; b < K; ++b)
      if (ranks_before(row[b], ids[p * K + b], row[best], ids[p * K + best])) best = b;
    double second = -kInf;
    for (int b = 0; b < K; ++b)
      if (b != best) second = std::max(second, row[b]);
    if (K > 1) mm = std::min(mm, rel(row[best] - second, row[best]));
    path[p] = ids[p * K + best];
    path_idx[p] = best;
    total += row[best];
    a = best;
  }
  *score = total;
  *margin = mm;
  return 0;
}

/* Viterbi max-sum, [ZhTW] §2 "Lightweight path selector (Path Selector)": one
 * dynamic-programming sweep finds the best path through the lattice.
 * delta_1(b) = S_1(x0,b); delta_t(b) = max_a [delta_{t-1}(a) + S_t(a,b)];
 * backtrack from argmax_b delta_{L-1}(b). Ties: lower token id, also for the
 * predecessor. margin = smallest relative best-vs-second gap among the
 * decisions on the returned path (final choice and each predecessor). */
int orc_path_viterbi(int P, int K, const double* S, const int32_t* ids, int32_t* path,
                     int32_t* path_idx, double* score, double* margin) {
  if (P < 1 || K < 1) return -1;
  std::vector<double> delta(K), next(K);
  std::vector<int> bp(static_cast<size_t>(P) * K, 0);
  std::vector<double> bm(static_cast<size_t>(P) * K, kInf);
  for (int b = 0; b < K; ++b) delta[b] = S[b];  // p = 0, a-row 0 holds S_1(x0, b)
  for (int p = 1; p < P; ++p) {
    for (int b = 0; b < K; ++b) {
      int best = 0;
      double bv = delta[0] + S[(static_cast<int64_t>(p) * K + 0) * K + b];
      double second = -kInf;
      for (int a = 1; a < K; ++a) {
        const double v = delta[a] + S[(static_cast<int64_t>(p) * K + a) * K + b];
        if (ranks_before(v, ids[(p - 1) * K + a], bv, ids[(p - 1) * K + best])) {
          second = std::max(second, bv);
          bv = v;
          best = a;
        } else {
          second = std::max(second, v);
        }
      }
      next[b] = bv;
      bp[p * K + b] = best;
      bm[p * K + b] = (K > 1) ? rel(bv - second, bv) : kInf;
    }
    delta.swap(next);
  }
  int fin = 0;
  for (int b = 1; b < K; ++b)
    if (ranks_before(delta[b], ids[(P - 1) * K + b], delta[fin], ids[(P - 1) * K + fin])) fin = b;
  double second = -kInf;
  for (int b = 0; b < K; ++b)
    if (b != fin) second = std::max(second, delta[b]);
  double mm = (K > 1) ? rel(delta[fin] - second, delta[fin]) : kInf;
  int cur = fin;
  for (int p = P - 1; p >= 0; --p) {
    path[p] = ids[p * K + cur];
    path_idx[p] = cur;
    if (p > 0) {
      mm = std::min(mm, bm[p * K + cur]);
      cur = bp[p * K + cur];
    }
  }
  *score = delta[fin];
  *margin = mm;
  return 0;
}

/* Greedy verification (T = 0), [ZhTW] §"The output is exactly the same" and
 * [Digest] §5: output identical to target-argmax decoding. Row i of Z is the
 * target's prediction after x_i (x_0 = last verified token), i = 0..L-1;
 * y_i = argmax_v Z[i][v]. n = largest k <= L-1 with x_t == y_{t-1} for all
 * t <= k. Emitted: x_1..x_n then y_n; accept_len = n + 1, which counts the
 * verifier's own next token as [Blog] Table 1's caption does. Unused output
 * slots are -1. */
int orc_verify_greedy(int zdtype, const void* Z, int L, int64_t V, const int32_t* path,
                      int32_t* out, int32_t* accept_len) {
  if (L < 2 || V < 1) return -1;
  std::vector<int64_t> y(L);
  for (int i = 0; i < L; ++i) {
    int64_t best = 0;
    double bv = widen(Z, zdtype, static_cast<int64_t>(i) * V);
    for (int64_t v = 1; v < V; ++v) {
      const double z = widen(Z, zdtype, static_cast<int64_t>(i) * V + v);
      if (z > bv) { bv = z; best = v; }
    }
    y[i] = best;
  }
  int n = 0;
  while (n < L - 1 && path[n] == y[n]) ++n;
  for (int i = 0; i < L; ++i) out[i] = -1;
  for (int i = 0; i < n; ++i) out[i] = path[i];
  out[n] = static_cast<int32_t>(y[n]);
  *accept_len = n + 1;
  return 0;
}

/* Rejection-sampling verification (T > 0), [Blog] §"A lightweight path
 * selector" (rejection sampling recovers the exact target distribution) and
 * [ZhTW] §"The output is exactly the same". The selected path is a
 * deterministic proposal. p_i = softmax(Z[i]/T). For t = 1..L-1: accept x_t
 * when U < p_{t-1}(x_t); on the first rejection emit a draw from p_{t-1}
 * with x_t removed and renormalised and stop (accept_len = t); when all are
 * accepted emit a bonus draw from p_{L-1} (accept_len = L). Each draw is redraw() above
 * with the position's one redraw uniform.
 * acc_margin = smallest |U - p| / p over the tests made; draw_margin = the
 * redraw's margin. b is the request's batch index (part of the counter). */
int orc_verify_sampling(int zdtype, const void* Z, int L, int64_t V, const int32_t* path,
                        double T, uint64_t seed, int64_t b, int32_t* out, int32_t* accept_len,
                        double* acc_margin, double* draw_margin) {
  if (L < 2 || V < 2 || !(T > 0.0)) return -1;
  for (int i = 0; i < L; ++i) out[i] = -1;
  double am = kInf;
  for (int t = 1; t < L; ++t) {
    const int64_t off = static_cast<int64_t>(t - 1) * V;
    const int64_t x = path[t - 1];
    const double p = std::exp(widen(Z, zdtype, off + x) / T - row_lse(Z, zdtype, off, V, T));
    const double u = uniform_accept(seed, b, t);
    am = std::min(am, std::fabs(u - p) / p);
    if (u < p) {
      out[t - 1] = static_cast<int32_t>(x);
      continue;
    }
    out[t - 1] = static_cast<int32_t>(
        redraw(Z, zdtype, off, V, T, uniform_redraw(seed, b, t), x, draw_margin));
    *accept_len = t;
    *acc_margin = am;
    return 0;
  }
  const int64_t off = static_cast<int64_t>(L - 1) * V;
  out[L - 1] = static_cast<int32_t>(
      redraw(Z, zdtype, off, V, T, uniform_redraw(seed, b, L), -1, draw_margin));
  *accept_len = L;
  *acc_margin = am;
  return 0;
}

/* The sampling verification above run once per seed in [seed0, seed0 + n), for
 * the distribution tests: out [n][L], accept_len [n]. */
int orc_verify_sampling_many(int zdtype, const void* Z, int L, int64_t V, const int32_t* path,
                             double T, uint64_t seed0, int64_t n, int64_t b, int nthreads,
                             int32_t* out, int32_t* accept_len) {
  if (L < 2 || V < 2 || !(T > 0.0) || n < 0) return -1;
  int bad = 0;
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads) reduction(| : bad)
  for (int64_t i = 0; i < n; ++i) {
    double am, gm;
    bad |= orc_verify_sampling(zdtype, Z, L, V, path, T, seed0 + static_cast<uint64_t>(i), b,
                               out + i * L, accept_len + i, &am, &gm);
  }
  return bad ? -1 : 0;
}

/* Sampled traversal, [Blog] §"A lightweight path selector": the same left-to-right
 * traversal from the last verified token as the greedy one, with each successor drawn from
 * the same scores instead of taken as the best: q_t(c) = softmax_c(S_t(x_{t-1}, c) / T)
 * over position t's K candidates, x_t drawn by one uniform against the cumulative q in
 * candidate order (if rounding leaves no candidate above it, the last one with mass).
 * Outputs the path, its candidate indices, q [P][K] (each position's distribution given
 * the drawn predecessor), the summed scores and the smallest distance of a uniform to a
 * cumulative boundary. T > 0. */
int orc_path_sample(int P, int K, const double* S, const int32_t* ids, double T, uint64_t seed,
                    int64_t b, int32_t* path, int32_t* pidx, double* q, double* score,
                    double* margin) {
  if (P < 1 || K < 1 || !(T > 0.0)) return -1;
  int a = 0;
  double total = 0.0, mg = kInf;
  for (int p = 0; p < P; ++p) {
    const double* row = S + (static_cast<int64_t>(p) * K + a) * K;
    double m = -kInf;
    for (int c = 0; c < K; ++c) m = std::max(m, row[c] / T);
    double z = 0.0;
    for (int c = 0; c < K; ++c) z += std::exp(row[c] / T - m);
    double* qp = q + static_cast<int64_t>(p) * K;
    for (int c = 0; c < K; ++c) qp[c] = std::exp(row[c] / T - m) / z;
    const double u = uniform_path(seed, b, p + 1);
    int pick = -1, last = 0;
    double cum = 0.0;
    for (int c = 0; c < K; ++c) {
      cum += qp[c];
      if (qp[c] > 0.0) last = c;
      if (c + 1 < K) mg = std::min(mg, std::fabs(cum - u));
      if (pick < 0 && cum > u) pick = c;
    }
    if (pick < 0) pick = last;
    path[p] = ids[static_cast<int64_t>(p) * K + pick];
    pidx[p] = pick;
    total += row[pick];
    a = pick;
  }
  *score = total;
  *margin = mg;
  return 0;
}

/* Joint path draw, [Blog] §"A lightweight path selector" (sampling draws from the same
 * scores), read as a draw of the whole path from the distribution the scores define over the
 * lattice: P(x_1..x_P) proportional to exp(sum_t S_t(x_{t-1}, x_t) / T), x_0 the last
 * verified token. Its conditionals come from backward messages
 *   log beta_P(c) = 0,  log beta_t(a) = log sum_c exp(S_{t+1}(a, c) / T + log beta_{t+1}(c)),
 * q_t(c | x_{t-1}) = exp(S_t(x_{t-1}, c) / T + log beta_t(c)) / (the same summed over c),
 * and x_t is drawn left to right from them, one uniform per position (counter (0, t, b, 3),
 * word 0) against the cumulative q in candidate order (if rounding leaves no candidate above
 * it, the last one with mass). Outputs as orc_path_sample: the path, its candidate indices,
 * q [P][K] (each position's conditional given the drawn predecessor), the summed scores and
 * the smallest distance of a uniform to a cumulative boundary. T > 0. */
int orc_path_sample_joint(int P, int K, const double* S, const int32_t* ids, double T,
                          uint64_t seed, int64_t b, int32_t* path, int32_t* pidx, double* q,
                          double* score, double* margin) {
  if (P < 1 || K < 1 || !(T > 0.0)) return -1;
  std::vector<double> lb(static_cast<size_t>(P) * K, 0.0);  // log beta_t, position t = p + 1
  for (int p = P - 2; p >= 0; --p) {
    for (int a = 0; a < K; ++a) {
      const double* row = S + (static_cast<int64_t>(p + 1) * K + a) * K;
      double m = -kInf;
      for (int c = 0; c < K; ++c) m = std::max(m, row[c] / T + lb[(p + 1) * K + c]);
      double z = 0.0;
      for (int c = 0; c < K; ++c) z += std::exp(row[c] / T + lb[(p + 1) * K + c] - m);
      lb[p * K + a] = m + std::log(z);
    }
  }
  int a = 0;
  double total = 0.0, mg = kInf;
  for (int p = 0; p < P; ++p) {
    const double* row = S + (static_cast<int64_t>(p) * K + a) * K;
    double m = -kInf;
    for (int c = 0; c < K; ++c) m = std::max(m, row[c] / T + lb[p * K + c]);
    double z = 0.0;
    for (int c = 0; c < K; ++c) z += std::exp(row[c] / T + lb[p * K + c] - m);
    double* qp = q + static_cast<int64_t>(p) * K;
    for (int c = 0; c < K; ++c) qp[c] = std::exp(row[c] / T + lb[p * K + c] - m) / z;
    const double u = uniform_path(seed, b, p + 1);
    int pick = -1, last = 0;
    double cum = 0.0;
    for (int c = 0; c < K; ++c) {
      cum += qp[c];
      if (qp[c] > 0.0) last = c;
      if (c + 1 < K) mg = std::min(mg, std::fabs(cum - u));
      if (pick < 0 && cum > u) pick = c;
    }
    if (pick < 0) pick = last;
    path[p] = ids[static_cast<int64_t>(p) * K + pick];
    pidx[p] = pick;
    total += row[pick];
    a = pick;
  }
  *score = total;
  *margin = mg;
  return 0;
}

/* Speculative-sampling verification of a sampled proposal, [Blog] §"A lightweight path
 * selector" (rejection sampling recovers the exact target distribution): for t = 1..L-1,
 * with p = softmax(Z[t-1]/T) and q = q_t (K candidates cand[t-1][*], the drawn one at index
 * pidx[t-1]): accept x_t when U < p(x_t) / q(x_t); on the first rejection emit a draw from
 * the residual max(0, p - q) renormalised and stop (accept_len = t); when all are accepted
 * emit a bonus draw from p_{L-1} (accept_len = L). Each emitted token is distributed as
 * p given the tokens before it (Leviathan, Kalman, Matias, ICML 2023; Chen et al. 2023).
 * A proposal that puts all its mass on x_t gives orc_verify_sampling. */
int orc_verify_proposal(int zdtype, const void* Z, int L, int64_t V, const int32_t* path,
                        const int32_t* cand, const double* q, const int32_t* pidx, int K, double T,
                        uint64_t seed, int64_t b, int32_t* out, int32_t* accept_len,
                        double* acc_margin, double* draw_margin) {
  if (L < 2 || V < 2 || K < 1 || !(T > 0.0)) return -1;
  for (int i = 0; i < L; ++i) out[i] = -1;
  double am = kInf;
  for (int t = 1; t < L; ++t) {
    const int64_t off = static_cast<int64_t>(t - 1) * V;
    const int64_t x = path[t - 1];
    const double p = std::exp(widen(Z, zdtype, off + x) / T - row_lse(Z, zdtype, off, V, T));
    const double qx = q[static_cast<int64_t>(t - 1) * K + pidx[t - 1]];
    const double ratio = p / qx;
    const double u = uniform_accept(seed, b, t);
    am = std::min(am, std::fabs(u - ratio) / ratio);
    if (u < ratio) {
      out[t - 1] = static_cast<int32_t>(x);
      continue;
    }
    out[t - 1] = static_cast<int32_t>(redraw_residual(Z, zdtype, off, V, T,
                                                      uniform_redraw(seed, b, t),
                                                      cand + static_cast<int64_t>(t - 1) * K,
                                                      q + static_cast<int64_t>(t - 1) * K, K,
                                                      draw_margin));
    *accept_len = t;
    *acc_margin = am;
    return 0;
  }
  const int64_t off = static_cast<int64_t>(L - 1) * V;
  out[L - 1] = static_cast<int32_t>(redraw_residual(Z, zdtype, off, V, T, uniform_redraw(seed, b, L),
                                                    nullptr, nullptr, 0, draw_margin));
  *accept_len = L;
  *acc_margin = am;
  return 0;
}

/* The sampled traversal (joint != 0: the joint path draw) and its verification run once per
 * seed in [seed0, seed0 + n) on a fixed lattice (S [P][K][K], ids [P][K]) and target rows
 * Z [L][V], for the distribution tests: paths [n][P], out [n][L], accept_len [n]. */
int orc_sample_verify_many(int zdtype, const void* Z, int L, int64_t V, const double* S,
                           const int32_t* ids, int K, double T, uint64_t seed0, int64_t n,
                           int64_t b, int nthreads, int joint, int32_t* paths, int32_t* out,
                           int32_t* accept_len) {
  if (L < 2 || V < 2 || K < 1 || !(T > 0.0) || n < 0) return -1;
  const int P = L - 1;
  int bad = 0;
  if (nthreads <= 0) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads) reduction(| : bad)
  for (int64_t i = 0; i < n; ++i) {
    std::vector<int32_t> pidx(P);
    std::vector<double> q(static_cast<size_t>(P) * K);
    double score, pm, am, gm;
    const uint64_t seed = seed0 + static_cast<uint64_t>(i);
    int rc = joint ? orc_path_sample_joint(P, K, S, ids, T, seed, b, paths + i * P, pidx.data(),
                                           q.data(), &score, &pm)
                   : orc_path_sample(P, K, S, ids, T, seed, b, paths + i * P, pidx.data(),
                                     q.data(), &score, &pm);
    if (rc == 0)
      rc = orc_verify_proposal(zdtype, Z, L, V, paths + i * P, ids, q.data(), pidx.data(), K, T,
                               seed, b, out + i * L, accept_len + i, &am, &gm);
    bad |= (rc != 0);
  }
  return bad ? -1 : 0;
}

/* The redraw of one target row Z [V] for given uniforms u [n] (instead of the counter's),
 * for the enumeration pins: K = 0 draws from softmax(z/T) with token excl removed (excl < 0:
 * none); K > 0 from the residual max(0, p - q) of the proposal cand [K] / qv [K] (excl is
 * then ignored). out [n] token ids, margin [n] as inverse_cdf's. */
int orc_redraw_uniforms(int zdtype, const void* Z, int64_t V, double T, int64_t excl,
                        const int32_t* cand, const double* qv, int K, const double* u, int64_t n,
                        int64_t* out, double* margin) {
  if (V < 1 || !(T > 0.0) || K < 0 || n < 0) return -1;
  for (int64_t i = 0; i < n; ++i)
    out[i] = K > 0 ? redraw_residual(Z, zdtype, 0, V, T, u[i], cand, qv, K, margin + i)
                   : redraw(Z, zdtype, 0, V, T, u[i], excl, margin + i);
  return 0;
}

/* Raw Philox4x64-10 block, exposed for the library pin. */
void orc_philox4x64(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  philox4x64_10(ctr, key, out);
}

/* The whole step for the listed requests of a batch, composed from the
 * stages above in the pages' order: logits -> keep top-K -> gate -> pair
 * scores -> path -> verify. Inputs: h [B][L][d], W [d][V], Wg [r][d],
 * A and Bt [V][r], x0 [B], Z [B][L][V]. Outputs are indexed by list position
 * q = 0..nreq-1. Wq / w_scale non-null: the LM head is E4M3 (orc_logits_e4m3) instead of W.
 * path_mode 0 = greedy traversal, 1 = Viterbi, 2 = sampled traversal, 3 = joint path draw
 * (2 and 3 verified against their own proposal); T <= 0 selects greedy verification (and,
 * for path_mode 2, the greedy traversal; for path_mode 3, Viterbi, the draw's T -> 0 limit). */
int orc_select_verify(int dtype, int zdtype, const void* h, const void* W, const void* Wg,
                      const void* A, const void* Bt, const int32_t* x0, const void* Z,
                      int64_t B, int L, int64_t V, int64_t d, int64_t r, int K, int path_mode,
                      double T, uint64_t seed, const int64_t* reqs, int64_t nreq, int nthreads,
                      int32_t* cand_ids, double* cand_U, double* gate, double* S, int32_t* path,
                      double* path_score, int32_t* out, int32_t* accept_len, double* topk_gap,
                      double* path_margin, double* acc_margin, double* draw_margin,
                      const uint8_t* Wq, const float* w_scale) {
  if (L < 2 || K < 1 || V < K || B < 1) return -1;
  const int P = L - 1;
  std::vector<int64_t> rows(P);
  std::vector<double> u(static_cast<size_t>(P) * V);
  std::vector<int32_t> pidx(P);
  for (int64_t q = 0; q < nreq; ++q) {
    const int64_t b = reqs[q];
    if (b < 0 || b >= B) return -1;
    for (int p = 0; p < P; ++p) rows[p] = b * L + (p + 1);
    int32_t* ids = cand_ids + q * P * K;
    double* U = cand_U + q * P * K;
    double* g = gate + q * P * r;
    double* Sq = S + q * P * K * K;
    int rc;
    if (Wq != nullptr) {  // E4M3 LM head: rows quantised, then the E4M3 product
      std::vector<uint8_t> hq(static_cast<size_t>(P) * d);
      std::vector<double> hs(P);
      rc = orc_quantize_rows_e4m3(dtype, h, d, rows.data(), P, hq.data(), hs.data());
      if (rc == 0)
        rc = orc_logits_e4m3(hq.data(), hs.data(), Wq, w_scale, d, V, P, u.data(), nthreads);
    } else {
      rc = orc_logits(dtype, h, W, d, V, rows.data(), P, u.data(), nthreads);
    }
    if (rc == 0) rc = orc_topk(u.data(), P, V, K, ids, U, topk_gap + q * P);
    if (rc == 0) rc = orc_gate(dtype, h, Wg, d, r, rows.data(), P, g);
    if (rc == 0) rc = orc_pair_scores(dtype, A, Bt, r, P, K, ids, U, g, x0[b], Sq);
    const bool sampled = (path_mode == 2 || path_mode == 3) && T > 0.0;
    std::vector<double> qprop(static_cast<size_t>(P) * K);
    if (rc == 0) {
      if (sampled && path_mode == 3)
        rc = orc_path_sample_joint(P, K, Sq, ids, T, seed, b, path + q * P, pidx.data(),
                                   qprop.data(), path_score + q, path_margin + q);
      else if (sampled)
        rc = orc_path_sample(P, K, Sq, ids, T, seed, b, path + q * P, pidx.data(), qprop.data(),
                             path_score + q, path_margin + q);
      else if (path_mode == 1 || path_mode == 3)
        rc = orc_path_viterbi(P, K, Sq, ids, path + q * P, pidx.data(), path_score + q, path_margin + q);
      else
        rc = orc_path_greedy(P, K, Sq, ids, path + q * P, pidx.data(), path_score + q, path_margin + q);
    }
    if (rc != 0) return rc;
    const char* zb = static_cast<const char*>(Z) +
                     b * static_cast<int64_t>(L) * V * (zdtype == ORC_BF16 ? 2 : 4);
    acc_margin[q] = kInf;
    draw_margin[q] = kInf;
    if (sampled)
      rc = orc_verify_proposal(zdtype, zb, L, V, path + q * P, ids, qprop.data(), pidx.data(), K,
                               T, seed, b, out + q * L, accept_len + q, acc_margin + q,
                               draw_margin + q);
    else if (T > 0.0)
      rc = orc_verify_sampling(zdtype, zb, L, V, path + q * P, T, seed, b, out + q * L,
                               accept_len + q, acc_margin + q, draw_margin + q);
    else
      rc = orc_verify_greedy(zdtype, zb, L, V, path + q * P, out + q * L, accept_len + q);
    if (rc != 0) return rc;
  }
  return 0;
}

/* Two-tap dynamic depthwise convolution, [Blog] §"A lightweight local convolution" (its
 * equation and Fig. 4): Conv_k(x)_t = k_{t,0} (.) x_t + k_{t,1} (.) x_{t-1} over the L
 * positions of each block, elementwise over the d channels. The pages give each coefficient
 * as a learned base kernel plus a small correction computed from the current hidden state,
 * one correction shared by every 16 channels, and say the first position reads the last
 * verified token. Readings taken (the correction's form is not printed):
 *   k_{t,j}[c] = base[j][c] + corr_t[j * (d/16) + c / 16],  corr_t = Wc x_t  (Wc: [d/8][d]),
 *   a linear map of the position's own hidden state: 2 d + 2 (d/16) d parameters per
 *   convolution, which over the 20 convolutions of a five-layer drafter of width 2560 (one
 *   before and after each attention and MLP sublayer) is the 16.5M the [Blog] reports;
 *   row 0 of a block is the last verified token, whose predecessor is outside the block;
 *   the convolution is block-local and stateless, so x_{-1} = 0 there.
 * x [nb][L][d] (xdtype), base [2][d] fp32, Wc [d/8][d] (wdtype); out [nb][L][d]. */
int orc_conv2tap(int xdtype, const void* x, const float* base, int wdtype, const void* Wc,
                 int64_t nb, int64_t L, int64_t d, double* out) {
  if (nb < 0 || L < 1 || d < 16 || d % 16 != 0) return -1;
  const int64_t G = d / 16;
  std::vector<double> corr(2 * G);
  for (int64_t b = 0; b < nb; ++b)
    for (int64_t t = 0; t < L; ++t) {
      const int64_t row = b * L + t;
      for (int64_t n = 0; n < 2 * G; ++n) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k) acc += widen(Wc, wdtype, n * d + k) * widen(x, xdtype, row * d + k);
        corr[n] = acc;
      }
      for (int64_t c = 0; c < d; ++c) {
        const double k0 = static_cast<double>(base[c]) + corr[c / 16];
        const double k1 = static_cast<double>(base[d + c]) + corr[G + c / 16];
        const double prev = t > 0 ? widen(x, xdtype, (row - 1) * d + c) : 0.0;
        out[row * d + c] = k0 * widen(x, xdtype, row * d + c) + k1 * prev;
      }
    }
  return 0;
}

}  // extern "C"
