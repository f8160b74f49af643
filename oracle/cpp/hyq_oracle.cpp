// Test infrastructure: a plain, slow CPU restatement of the hybrid-precision
// attention method of "HyQuant: Hybrid-Precision Quantization for LLM
// Attention", in float64, for checking the CUDA library against.  Nothing
// here is shared with the kernels: the number formats are written from
// their definitions, every step follows the paper's order, and only the
// tests and the benchmark's CPU-baseline legs load this library.
//
//   quantiser        Appendix A.4 Algorithm 4 (Quant_B), Eq. 9 (DeQuant)
//   selection        Appendix A.1 Algorithm 1 (summed proxy logits), per KV
//                    head and per query head (its B x H_Q x k output, kept
//                    per KV head as the union filled by the group score),
//                    and the softmax-mass score of §4.1 Eq. 4 with Eq. 5's
//                    top-k
//   decode           §4.3 Eq. 8-9: softmax attention over the effective cache
//   prefill          §4.2 Eq. 6-7, Appendix A.2 Algorithm 2
//
// Readings where the paper is silent (one line each; the same as the Python
// oracle): groups of 32 along head_dim; x ~ c s + z with s the smallest
// binary16 step covering the group's range and z = RN_binary16(min); codes
// are the nearest grid point, ties to even; one vertical-line set per KV
// head with ties to the lower position (per query head: the union of a
// group's sets filled up to min(P, g k) by the group score); prefill scales
// s = RN_binary32(max|x| / c_B) per 64-key tile and per 128-row query block,
// codes the grid value nearest to the exact quotient x / s (INT8, e4m3 or
// e2m1 with c_B = 127, 448, 6).
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -shared -fPIC (no fused
// multiply-add may change a rounding; every operation is one IEEE double
// operation).  All entry points take float64 arrays whose values are exactly
// representable in BF16 (the inputs of the method) and are thread-safe.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <functional>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits;
// the spacing of its numbers at magnitude a > 0 is 2^(max(e, -14) - 10) where
// 2^e <= a < 2^(e+1); the largest finite value is 65504.
double fp16_spacing(double a) {
  int e2 = 0;
  std::frexp(a, &e2);  // a = f 2^e2, f in [0.5, 1): leading bit 2^(e2 - 1)
  return std::ldexp(1.0, std::max(e2 - 1, -14) - 10);
}

// Nearest binary16 value to x, ties to even; +-inf beyond the range.
double fp16_rn(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  const double a = std::fabs(x), q = fp16_spacing(a);
  const double r = std::nearbyint(a / q) * q;  // a / q and the product are exact
  const double out = r > 65504.0 ? INFINITY : r;
  return x < 0 ? -out : out;
}

// Smallest binary16 value >= x, for x >= 0.
double fp16_ru(double x) {
  if (x <= 0.0) return 0.0;
  const double q = fp16_spacing(x);
  const double r = std::ceil(x / q) * q;
  return r > 65504.0 ? INFINITY : r;
}

// The binary16 values adjacent to a positive binary16 value h.
double fp16_next_up(double h) { return h == 0.0 ? std::ldexp(1.0, -24) : h + fp16_spacing(h); }
double fp16_next_down(double h) {
  int e2 = 0;
  const double f = std::frexp(h, &e2);
  const double q = fp16_spacing(h);
  return (f == 0.5 && e2 - 1 > -14) ? h - q / 2 : h - q;  // below a power of two the spacing halves
}

// e4m3 (the "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
// bits; exponent field 0 holds subnormals m 2^-9; exponent 15 with fraction 7
// is NaN and there are no infinities, so the largest value is 448.  The
// non-negative values in ascending order; an index is the 7-bit code.
std::vector<double> e4m3_values() {
  std::vector<double> v;
  for (int e = 0; e < 16; ++e)
    for (int m = 0; m < 8; ++m) {
      if (e == 15 && m == 7) continue;
      v.push_back(e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7));
    }
  return v;
}

// e2m1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; exponent
// field 0 holds the subnormal m 2^-1; no infinities or NaN, so the largest
// value is 6.  The non-negative values in ascending order (index = code).
std::vector<double> e2m1_values() {
  std::vector<double> v;
  for (int e = 0; e < 4; ++e)
    for (int m = 0; m < 2; ++m) v.push_back(e == 0 ? m * 0.5 : (1.0 + m / 2.0) * std::ldexp(1.0, e - 1));
  return v;
}

// ---------------------------------------------------------------------------
// Exact arithmetic helpers
// ---------------------------------------------------------------------------

// a + b = s + e exactly (error-free transformation; no overflow assumed).
void two_sum(double a, double b, double& s, double& e) {
  s = a + b;
  const double bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Sign of the exact sum of a few doubles: the terms are accumulated into a
// nonoverlapping expansion (components of increasing magnitude), whose sign
// is that of its largest component.
int sign_of_sum(std::initializer_list<double> terms) {
  std::vector<double> ex;
  for (double t : terms) {
    std::vector<double> h;
    double q = t;
    for (double e : ex) {
      double s, err;
      two_sum(q, e, s, err);
      if (err != 0.0) h.push_back(err);
      q = s;
    }
    if (q != 0.0) h.push_back(q);
    ex.swap(h);
  }
  for (auto it = ex.rbegin(); it != ex.rend(); ++it)
    if (*it != 0.0) return *it > 0.0 ? 1 : -1;
  return 0;
}

// Runs f(i) for i in [0, n) on `threads` workers (0: every hardware thread).
void parallel_for(int64_t n, int threads, const std::function<void(int64_t)>& f) {
  int nt = threads > 0 ? threads : (int)std::max(1u, std::thread::hardware_concurrency());
  nt = (int)std::min<int64_t>(nt, std::max<int64_t>(n, 1));
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int w = 0; w < nt; ++w)
    pool.emplace_back([&] {
      for (int64_t i = next++; i < n; i = next++) f(i);
    });
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------------------
// Algorithm 4 Quant_B, Eq. 9 DeQuant
// ---------------------------------------------------------------------------

// The smallest binary16 h with qmax h >= mx - mn in exact arithmetic.
double min_step(double mx, double mn, int qmax) {
  auto covers = [&](double h) { return sign_of_sum({qmax * h, -mx, mn}) >= 0; };  // qmax h is exact
  double h = fp16_ru((mx - mn) / qmax);
  if (!std::isfinite(h)) return h;
  while (h > 0.0 && covers(fp16_next_down(h))) h = fp16_next_down(h);
  while (!covers(h)) h = fp16_next_up(h);
  return h;
}

// Index c in [0, qmax] of the grid point z + c s nearest to x, ties to the
// even index.  Each midpoint z + (c +- 1/2) s is exact in float64 (s and z
// are binary16: a multiple of 2^-25 below 2^25 in magnitude) and the sign of
// x minus it is exact, so the candidate from a float64 quotient is corrected
// exactly.
int nearest_code(double x, double z, double s, int qmax) {
  if (!(s > 0.0)) return 0;
  double c = std::min<double>(std::max(std::nearbyint((x - z) / s), 0.0), qmax);
  for (int it = 0; it < 2; ++it) {
    if (c < qmax) {
      const double d = x - (z + (c + 0.5) * s);
      if (d > 0.0 || (d == 0.0 && std::fmod(c, 2.0) == 1.0)) c += 1.0;
    }
    if (c > 0) {
      const double d = x - (z + (c - 0.5) * s);
      if (d < 0.0 || (d == 0.0 && std::fmod(c, 2.0) == 1.0)) c -= 1.0;
    }
  }
  return (int)c;
}

// Quantise one row of d elements (d a multiple of 32): codes, per-group step
// and zero.  Returns false if a step or zero is not a finite binary16.
bool quantize_row(const double* x, int d, int bits, uint8_t* codes, double* scale, double* zero) {
  const int qmax = (1 << bits) - 1;
  bool ok = true;
  for (int g = 0; g < d / 32; ++g) {
    const double* xg = x + 32 * g;
    double mn = xg[0], mx = xg[0];
    for (int i = 1; i < 32; ++i) {
      mn = std::min(mn, xg[i]);
      mx = std::max(mx, xg[i]);
    }
    const double s = min_step(mx, mn, qmax), z = fp16_rn(mn);
    if (!std::isfinite(s) || !std::isfinite(z) || std::isnan(mn) || std::isnan(mx)) ok = false;
    scale[g] = s;
    zero[g] = z;
    for (int i = 0; i < 32; ++i) codes[32 * g + i] = (uint8_t)nearest_code(xg[i], z, s, qmax);
  }
  return ok;
}

// DeQuant(Quant(row)) in place into out.
bool fake_quant_row(const double* x, int d, int bits, double* out) {
  std::vector<uint8_t> c(d);
  std::vector<double> s(d / 32), z(d / 32);
  const bool ok = quantize_row(x, d, bits, c.data(), s.data(), z.data());
  for (int i = 0; i < d; ++i) out[i] = c[i] * s[i / 32] + z[i / 32];
  return ok;
}

// ---------------------------------------------------------------------------
// Algorithm 1 (and Eq. 4-5)
// ---------------------------------------------------------------------------

int64_t vl_count(int64_t P, int64_t rho_ppm) {
  if (P <= 0 || rho_ppm <= 0) return 0;
  const int64_t k = (P * rho_ppm + 999999) / 1000000;  // exact ceil(P rho)
  return std::min(P, std::max<int64_t>(1, k));
}

// Top-k of S[0..P) by (score descending, position ascending), returned ascending.
void topk_ascending(const std::vector<double>& S, int64_t k, int64_t* out) {
  std::vector<int64_t> ord(S.size());
  for (size_t j = 0; j < S.size(); ++j) ord[j] = (int64_t)j;
  std::sort(ord.begin(), ord.end(), [&](int64_t a, int64_t b) { return S[a] > S[b] || (S[a] == S[b] && a < b); });
  std::sort(ord.begin(), ord.begin() + k);
  std::copy(ord.begin(), ord.begin() + k, out);
}

// ---------------------------------------------------------------------------
// Prefill codes (Algorithm 2 stage 2)
// ---------------------------------------------------------------------------

// Index into the ascending non-negative grid of the value nearest to the
// exact quotient a / s (a >= 0, s > 0), ties to the even index, values past
// the top taking the top; each midpoint times s is exact in float64.
int nearest_grid_index(double a, double s, const std::vector<double>& grid) {
  const int n = (int)grid.size() - 1;  // number of midpoints
  auto mid = [&](int i) { return (grid[i] + grid[i + 1]) / 2; };
  int i = 0;
  {
    const double qq = a / s;  // candidate: midpoints below the float64 quotient
    int lo = 0, hi = n;
    while (lo < hi) {
      const int m = (lo + hi) / 2;
      if (mid(m) < qq) lo = m + 1;
      else hi = m;
    }
    i = lo;
  }
  for (int it = 0; it < 2; ++it) {
    if (i < n) {
      const double d = a - mid(i) * s;
      if (d > 0.0 || (d == 0.0 && i % 2 == 1)) ++i;
    }
    if (i > 0) {
      const double d = a - mid(i - 1) * s;
      if (d < 0.0 || (d == 0.0 && i % 2 == 1)) --i;
    }
  }
  return i;
}

struct SymQuant {
  std::vector<double> grid;
  float cb;
  explicit SymQuant(int dtype) {
    if (dtype == 2) {
      grid = e4m3_values();
      cb = 448.f;
    } else if (dtype == 3) {
      grid = e2m1_values();
      cb = 6.f;
    } else {
      for (int i = 0; i < 128; ++i) grid.push_back(i);
      cb = 127.f;
    }
  }
  // Dequantised values of n elements with one scale s = RN_binary32(max|x| / c_B).
  void fake(const double* x, int64_t n, double* out) const {
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[i]));
    const float s32 = (float)amax / cb;  // one binary32 division (max|x| is exact in binary32)
    const double s = s32;
    for (int64_t i = 0; i < n; ++i) {
      if (!(s > 0.0)) {
        out[i] = 0.0;
        continue;
      }
      const double c = grid[nearest_grid_index(std::fabs(x[i]), s, grid)];
      out[i] = (x[i] < 0 ? -c : c) * s;
    }
  }
};

}  // namespace

extern "C" {

// Quantise n_rows rows of d elements (bits 4 or 8): codes [n_rows][d],
// scale and zero [n_rows][d / 32].  Returns 0, or 1 if a group's step or
// zero is not a finite binary16 (or the input holds a NaN).
int hyqo_quantize(const double* x, int64_t n_rows, int d, int bits, uint8_t* codes, double* scale, double* zero) {
  int bad = 0;
  for (int64_t r = 0; r < n_rows; ++r)
    if (!quantize_row(x + r * d, d, bits, codes + r * d, scale + r * (d / 32), zero + r * (d / 32))) bad = 1;
  return bad;
}

int64_t hyqo_vl_count(int64_t P, int64_t rho_ppm) { return vl_count(P, rho_ppm); }

// The e4m3 value of a 7-bit magnitude code (0 .. 126).
double hyqo_e4m3_value(int code) {
  static const std::vector<double> v = e4m3_values();
  return (code >= 0 && code < (int)v.size()) ? v[code] : NAN;
}

// The e2m1 value of a 3-bit magnitude code (0 .. 7).
double hyqo_e2m1_value(int code) {
  static const std::vector<double> v = e2m1_values();
  return (code >= 0 && code < (int)v.size()) ? v[code] : NAN;
}

// Vertical-line selection per (b, KV head).  q_proxy [B][HQ][T][d], k [B][HKV][ldk][d]
// (rows 0..L-1 used).  mass = 0: Algorithm 1's S(j) = u . k_j with u the sum
// of the T proxies over the g query heads of the KV head; mass = 1: Eq. 4's
// S(j) = sum over those T g rows of softmax over the L keys of
// (q . k_j / sqrt(d)).  Top-k over j < P = max(0, L - W), k = ceil(P rho)
// clamped to [1, P] (0 when P = 0 or rho = 0).  idx_out [B][HKV][k]
// ascending; scores_out [B][HKV][P] (may be null).  Returns k.
int64_t hyqo_select(const double* qp, const double* k, int B, int HQ, int HKV, int T, int64_t ldk, int d,
                    int64_t L, int64_t W, int64_t rho_ppm, int mass, int64_t* idx_out, double* scores_out,
                    int threads) {
  const int64_t P = std::max<int64_t>(0, L - W), kk = vl_count(P, rho_ppm);
  const int g = HQ / HKV;
  parallel_for((int64_t)B * HKV, threads, [&](int64_t bh) {
    const int64_t b = bh / HKV, kh = bh % HKV;
    const double* K = k + (b * HKV + kh) * ldk * d;
    std::vector<double> S(P, 0.0);
    if (!mass) {
      std::vector<double> u(d, 0.0);
      for (int h = 0; h < g; ++h)
        for (int t = 0; t < T; ++t) {
          const double* qr = qp + (((b * HQ) + kh * g + h) * (int64_t)T + t) * d;
          for (int i = 0; i < d; ++i) u[i] += qr[i];
        }
      for (int64_t j = 0; j < P; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += u[i] * K[j * d + i];
        S[j] = acc;
      }
    } else {
      const double alpha = 1.0 / std::sqrt((double)d);
      std::vector<double> z(L);
      for (int h = 0; h < g; ++h)
        for (int t = 0; t < T; ++t) {
          const double* qr = qp + (((b * HQ) + kh * g + h) * (int64_t)T + t) * d;
          double m = -INFINITY;
          for (int64_t j = 0; j < L; ++j) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += qr[i] * K[j * d + i];
            z[j] = alpha * acc;
            m = std::max(m, z[j]);
          }
          double l = 0.0;
          for (int64_t j = 0; j < L; ++j) l += std::exp(z[j] - m);
          for (int64_t j = 0; j < P; ++j) S[j] += std::exp(z[j] - m) / l;
        }
    }
    topk_ascending(S, kk, idx_out + bh * kk);
    if (scores_out) std::copy(S.begin(), S.end(), scores_out + bh * P);
  });
  return kk;
}

// Algorithm 1 per query head: S_h(j) = u_h . k_j with u_h the sum of query
// head h's T proxies and k_j the key of its KV head; each head keeps its k
// largest (ties to the lower position).  Per KV head the stored list is the
// union of its g heads' sets, filled up to ku = min(P, g k) positions with
// the largest group scores (Algorithm 1's per-KV-head S) among the others,
// ties to the lower position.  idx_heads [B][HQ][k], idx_kv [B][HKV][ku]
// (both ascending), union_size [B][HKV].  Returns ku.
int64_t hyqo_select_heads(const double* qp, const double* k, int B, int HQ, int HKV, int T, int64_t ldk, int d,
                          int64_t L, int64_t W, int64_t rho_ppm, int64_t* idx_heads, int64_t* idx_kv,
                          int64_t* union_size, int threads) {
  const int64_t P = std::max<int64_t>(0, L - W), kk = vl_count(P, rho_ppm);
  const int g = HQ / HKV;
  const int64_t ku = std::min<int64_t>(P, g * kk);
  parallel_for((int64_t)B * HKV, threads, [&](int64_t bh) {
    const int64_t b = bh / HKV, kh = bh % HKV;
    const double* K = k + (b * HKV + kh) * ldk * d;
    std::vector<double> Sg(P, 0.0), Sh(P);
    std::vector<char> in_union(std::max<int64_t>(P, 1), 0);
    std::vector<double> ug(d, 0.0);
    for (int h = 0; h < g; ++h) {
      std::vector<double> u(d, 0.0);
      for (int t = 0; t < T; ++t) {
        const double* qr = qp + (((b * HQ) + kh * g + h) * (int64_t)T + t) * d;
        for (int i = 0; i < d; ++i) u[i] += qr[i];
      }
      for (int i = 0; i < d; ++i) ug[i] += u[i];
      for (int64_t j = 0; j < P; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += u[i] * K[j * d + i];
        Sh[j] = acc;
      }
      int64_t* own = idx_heads + ((b * HQ) + kh * g + h) * kk;
      topk_ascending(Sh, kk, own);
      for (int64_t i = 0; i < kk; ++i) in_union[own[i]] = 1;
    }
    // the group score, with the proxies of all g heads summed first (as Algorithm 1 per KV head)
    for (int64_t j = 0; j < P; ++j) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += ug[i] * K[j * d + i];
      Sg[j] = acc;
    }
    int64_t nu = 0;
    for (int64_t j = 0; j < P; ++j) nu += in_union[j];
    union_size[bh] = nu;
    // fill: the positions outside the union by (group score descending, position ascending)
    std::vector<int64_t> rest;
    for (int64_t j = 0; j < P; ++j)
      if (!in_union[j]) rest.push_back(j);
    std::stable_sort(rest.begin(), rest.end(), [&](int64_t a, int64_t c) { return Sg[a] > Sg[c]; });
    for (int64_t i = 0; i < ku - nu && i < (int64_t)rest.size(); ++i) in_union[rest[i]] = 1;
    int64_t o = 0;
    for (int64_t j = 0; j < P; ++j)
      if (in_union[j]) idx_kv[bh * ku + o++] = j;
  });
  return ku;
}

// Hybrid decode attention (Eq. 8-9): for every query head h (KV head h / g)
//   o_h = sum_j exp(a q_h . k~_j - M) v~_j / sum_j exp(a q_h . k~_j - M), a = 1/sqrt(d),
// over j < L, with k~_j, v~_j = DeQuant(Quant(.)) (B_K / B_V bits) for j in
// [0, P) outside the vertical-line set idx, and the given rows otherwise.
// q [B][HQ][d]; k, v [B][HKV][ldk][d]; idx [B][HKV][kvl]; out [B][HQ][d].
// Returns 0, or 1 if some group was out of the binary16 range.
int hyqo_decode(const double* q, const double* k, const double* v, int B, int HQ, int HKV, int64_t ldk, int d,
                int64_t L, int64_t P, const int64_t* idx, int64_t kvl, int bits_k, int bits_v, double* out,
                int threads) {
  const int g = HQ / HKV;
  const double alpha = 1.0 / std::sqrt((double)d);
  std::atomic<int> bad{0};
  parallel_for((int64_t)B * HKV, threads, [&](int64_t bh) {
    const int64_t b = bh / HKV, kh = bh % HKV;
    const double* K = k + bh * ldk * d;
    const double* V = v + bh * ldk * d;
    std::vector<char> keep(std::max<int64_t>(P, 1), 0);
    for (int64_t i = 0; i < kvl; ++i)
      if (idx[bh * kvl + i] >= 0 && idx[bh * kvl + i] < P) keep[idx[bh * kvl + i]] = 1;
    std::vector<double> Ke(L * d), Ve(L * d);
    for (int64_t j = 0; j < L; ++j) {
      if (j < P && !keep[j]) {
        if (!fake_quant_row(K + j * d, d, bits_k, &Ke[j * d])) bad = 1;
        if (!fake_quant_row(V + j * d, d, bits_v, &Ve[j * d])) bad = 1;
      } else {
        std::copy(K + j * d, K + (j + 1) * d, &Ke[j * d]);
        std::copy(V + j * d, V + (j + 1) * d, &Ve[j * d]);
      }
    }
    std::vector<double> lg(L);
    for (int h = 0; h < g; ++h) {
      const double* qh = q + (b * HQ + kh * g + h) * (int64_t)d;
      double* oh = out + (b * HQ + kh * g + h) * (int64_t)d;
      double M = -INFINITY;
      for (int64_t j = 0; j < L; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += qh[i] * Ke[j * d + i];
        lg[j] = alpha * acc;
        M = std::max(M, lg[j]);
      }
      double den = 0.0;
      std::fill(oh, oh + d, 0.0);
      for (int64_t j = 0; j < L; ++j) {
        const double w = std::exp(lg[j] - M);
        den += w;
        for (int i = 0; i < d; ++i) oh[i] += w * Ve[j * d + i];
      }
      for (int i = 0; i < d; ++i) oh[i] /= den;
    }
  });
  return bad.load();
}

// Hybrid prefill (Eq. 7, Algorithm 2), causal.  q [B][HQ][L][d]; k, v
// [B][HKV][L][d]; idx [B][HKV][kvl] ascending in [0, P), P = max(0, L - W).
// The quantised prefix [0, P) minus idx, in ascending order, is cut into
// tiles of 64 keys, each with one scale for K and one for V; queries use
// one scale per 128-row block of one head; dtype 1 = INT8 (codes -127..127),
// 2 = FP8 e4m3, 3 = FP4 e2m1.  Quantised keys meet the quantised query, the others
// (vertical lines and, for band = 0, [P, L); for band = 1 the keys (i - W, i]
// of row i) the BF16 query; every key at or before the row (band = 1: the
// quantised prefix and vertical lines only at or before i - W).
// block_mask [ceil(L / 128)] and head_mask [HQ] (null = all) choose the
// rows computed; out and mag [B][HQ][L][d] (mag = sum_j p_j |v_j| / sum p).
void hyqo_prefill(const double* q, const double* k, const double* v, int B, int HQ, int HKV, int64_t L, int d,
                  int64_t W, const int64_t* idx, int64_t kvl, int dtype, int band, const uint8_t* block_mask,
                  const uint8_t* head_mask, double* out, double* mag, int threads) {
  const int g = HQ / HKV;
  const double alpha = 1.0 / std::sqrt((double)d);
  const int64_t P = std::max<int64_t>(0, L - W);
  const int64_t nblk = (L + 127) / 128;
  const SymQuant sq(dtype);
  // per (b, KV head): the effective key / value lists
  struct Lists {
    std::vector<int64_t> pos;     // positions of the quantised list, then the full-precision list
    std::vector<double> K, V;     // rows of both lists
    int64_t nq = 0;
  };
  std::vector<Lists> lists((size_t)B * HKV);
  parallel_for((int64_t)B * HKV, threads, [&](int64_t bh) {
    Lists& ls = lists[bh];
    const double* Kb = k + bh * L * d;
    const double* Vb = v + bh * L * d;
    std::vector<char> isvl(std::max<int64_t>(P, 1), 0);
    for (int64_t i = 0; i < kvl; ++i) isvl[idx[bh * kvl + i]] = 1;
    for (int64_t j = 0; j < P; ++j)
      if (!isvl[j]) ls.pos.push_back(j);
    ls.nq = (int64_t)ls.pos.size();
    for (int64_t i = 0; i < kvl; ++i) ls.pos.push_back(idx[bh * kvl + i]);
    if (!band)
      for (int64_t j = P; j < L; ++j) ls.pos.push_back(j);
    const int64_t n = (int64_t)ls.pos.size();
    ls.K.assign(n * d, 0.0);
    ls.V.assign(n * d, 0.0);
    std::vector<double> tk, tv;
    for (int64_t t0 = 0; t0 < ls.nq; t0 += 64) {  // quantised tiles
      const int64_t m = std::min<int64_t>(64, ls.nq - t0);
      tk.assign(m * d, 0.0);
      tv.assign(m * d, 0.0);
      for (int64_t r = 0; r < m; ++r) {
        std::copy(Kb + ls.pos[t0 + r] * d, Kb + (ls.pos[t0 + r] + 1) * d, &tk[r * d]);
        std::copy(Vb + ls.pos[t0 + r] * d, Vb + (ls.pos[t0 + r] + 1) * d, &tv[r * d]);
      }
      sq.fake(tk.data(), m * d, &ls.K[t0 * d]);
      sq.fake(tv.data(), m * d, &ls.V[t0 * d]);
    }
    for (int64_t r = ls.nq; r < n; ++r) {
      std::copy(Kb + ls.pos[r] * d, Kb + (ls.pos[r] + 1) * d, &ls.K[r * d]);
      std::copy(Vb + ls.pos[r] * d, Vb + (ls.pos[r] + 1) * d, &ls.V[r * d]);
    }
  });
  parallel_for((int64_t)B * HQ * nblk, threads, [&](int64_t item) {
    const int64_t b = item / (HQ * nblk), h = (item / nblk) % HQ, blk = item % nblk;
    if ((head_mask && !head_mask[h]) || (block_mask && !block_mask[blk])) return;
    const int64_t kh = h / g, bh = b * HKV + kh;
    const Lists& ls = lists[bh];
    const double* Kb = k + bh * L * d;
    const double* Vb = v + bh * L * d;
    const int64_t r0 = 128 * blk, r1 = std::min(L, r0 + 128);
    const double* qb = q + ((b * HQ + h) * L + r0) * d;
    std::vector<double> qhat((r1 - r0) * d);
    sq.fake(qb, (r1 - r0) * d, qhat.data());
    const int64_t n = (int64_t)ls.pos.size();
    std::vector<double> lg, wv;
    std::vector<const double*> vrow;
    for (int64_t i = r0; i < r1; ++i) {
      const double* qi = qb + (i - r0) * d;
      const double* qh = &qhat[(i - r0) * d];
      lg.clear();
      vrow.clear();
      const int64_t lim = band ? i - W : i;  // keys of both lists must lie at or before this
      for (int64_t r = 0; r < n; ++r) {
        if (ls.pos[r] > lim) continue;
        const double* qq = r < ls.nq ? qh : qi;
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += qq[e] * ls.K[r * d + e];
        lg.push_back(alpha * acc);
        vrow.push_back(&ls.V[r * d]);
      }
      if (band)
        for (int64_t j = std::max<int64_t>(0, i - W + 1); j <= i; ++j) {  // the band (i - W, i]
          double acc = 0.0;
          for (int e = 0; e < d; ++e) acc += qi[e] * Kb[j * d + e];
          lg.push_back(alpha * acc);
          vrow.push_back(Vb + j * d);
        }
      double M = -INFINITY;
      for (double x : lg) M = std::max(M, x);
      double den = 0.0;
      double* o = out + ((b * HQ + h) * L + i) * d;
      double* ma = mag ? mag + ((b * HQ + h) * L + i) * d : nullptr;
      std::fill(o, o + d, 0.0);
      if (ma) std::fill(ma, ma + d, 0.0);
      for (size_t r = 0; r < lg.size(); ++r) {
        const double w = std::exp(lg[r] - M);
        den += w;
        for (int e = 0; e < d; ++e) {
          o[e] += w * vrow[r][e];
          if (ma) ma[e] += w * std::fabs(vrow[r][e]);
        }
      }
      for (int e = 0; e < d; ++e) {
        o[e] /= den;
        if (ma) ma[e] /= den;
      }
    }
  });
}

}  // extern "C"
