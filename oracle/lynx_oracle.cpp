// Plain C++ CPU oracle of the RT-Lynx activation-sparse linear layer.
//
// TEST INFRASTRUCTURE.  Only the tests, __graft_entry__.smoke() and the CPU
// arms of bench.py (the timed CPU baseline and --impl reference) load this
// library, through oracle/cpp.py.  The CUDA library never does, and the two
// share no code: this file includes nothing but the C++ standard library.
//
// What is computed follows the RT-Lynx page (aitrends.kr article 60737):
//
//   Method, "key mechanism": a Top-K based 2:4 selection of the activations
//     gives X~; the sparse activation is S(X) = s * X~; the output is
//     Y = Ys + Yr with Ys = S(X) W^T and Yr = X (LA LB)^T.
//   Code examples, first formula: s = ||X||_2 / (||X~||_2 + eps), which
//     restores the dense activation's L2 norm (Glossary, "Norm Compensation").
//   Technical details: LoRA rank 64; selected single-stream layers are left
//     dense (Selective Layer Skipping).
//   Main results / Key idea: the "Sparse Weight" comparator (2:4 pruning of W).
//
// Readings taken where the page is silent:
//   - a group is 4 consecutive input channels (the K axis) of one token row;
//   - "top-K" keeps the two largest |x| of a group; ties go to the lower index
//     (a stable sort by |x|, largest first); a group with fewer than two
//     nonzeros still keeps exactly two positions;
//   - the norm is per token over all K channels; eps = 0, and a row whose kept
//     entries are all zero has s = 1;
//   - the LoRA branch takes the dense, unscaled X and is evaluated as
//     (X LB^T) LA^T, the same product as X (LA LB)^T;
//   - no bias; results are returned in double (the CUDA path rounds Y to bf16);
//   - the weight-2:4 comparator keeps the two largest |w| of every 4
//     consecutive input channels of each row of W, ties to the lower index,
//     with no norm compensation.
//
// Everything is double precision computed from the bf16 inputs (uint16 bit
// patterns, row-major: X M x K, W N x K, LA N x R, LB R x K).  Sums run over
// their index in increasing order; there is no blocking, tiling or fusion.
// Rows are independent, so the row loop is split over T std::threads; the
// result does not depend on T.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

double widen_one(uint16_t b) {
  // a bf16 value is the upper half of an IEEE binary32 value
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return static_cast<double>(f);
}

std::vector<double> widen_all(const uint16_t* bits, int64_t n) {
  std::vector<double> out(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) out[static_cast<size_t>(i)] = widen_one(bits[i]);
  return out;
}

// Runs body(i) for i in [0, n) on `threads` std::threads, each taking one contiguous range.
void parallel_rows(int64_t n, int threads, const std::function<void(int64_t)>& body) {
  if (threads < 1) threads = static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  if (threads > n) threads = static_cast<int>(std::max<int64_t>(n, 1));
  if (threads <= 1) {
    for (int64_t i = 0; i < n; ++i) body(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(static_cast<size_t>(threads));
  for (int t = 0; t < threads; ++t) {
    const int64_t lo = n * t / threads, hi = n * (t + 1) / threads;
    pool.emplace_back([lo, hi, &body] {
      for (int64_t i = lo; i < hi; ++i) body(i);
    });
  }
  for (auto& th : pool) th.join();
}

// The kept pair of one group of four (RT-Lynx page, Method: Top-K based 2:4 selection): the four positions
// ordered by |x|, largest first, by a stable sort (so of two equal magnitudes the lower position comes
// first); the first two positions of that order, returned in increasing order.
void select_group(const double* g, int* i0, int* i1) {
  int order[4] = {0, 1, 2, 3};
  std::stable_sort(order, order + 4, [g](int a, int b) { return std::fabs(g[a]) > std::fabs(g[b]); });
  *i0 = std::min(order[0], order[1]);
  *i1 = std::max(order[0], order[1]);
}

// keep[k] = 1 for the two kept positions of every group of the row.
void keep_row(const double* x, int64_t K, uint8_t* keep) {
  for (int64_t g = 0; g < K / 4; ++g) {
    int i0, i1;
    select_group(x + 4 * g, &i0, &i1);
    for (int j = 0; j < 4; ++j) keep[4 * g + j] = (j == i0 || j == i1) ? 1 : 0;
  }
}

// s = sqrt(sum x^2 / sum x~^2) (Code examples, first formula, eps = 0); 1 when the kept entries are all zero.
double scale_row(const double* x, const uint8_t* keep, int64_t K) {
  double nx = 0.0, nt = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    nx += x[k] * x[k];
    if (keep[k]) nt += x[k] * x[k];
  }
  return nt > 0.0 ? std::sqrt(nx / nt) : 1.0;
}

// Row m of the LoRA branch X (LA LB)^T, as (X LB^T) LA^T: t[r] = sum_k x_k LB[r,k], then yr[n] = sum_r t[r] LA[n,r].
void lora_row(const double* x, const double* la, const double* lb, int64_t N, int64_t K, int64_t R, double* yr) {
  std::vector<double> t(static_cast<size_t>(R), 0.0);
  for (int64_t r = 0; r < R; ++r) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += x[k] * lb[r * K + k];
    t[static_cast<size_t>(r)] = acc;
  }
  for (int64_t n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int64_t r = 0; r < R; ++r) acc += t[static_cast<size_t>(r)] * la[n * R + r];
    yr[n] = acc;
  }
}

// y[n] = sum_k a[k] W[n,k]: one output row of a product with W^T.
void product_row(const double* a, const double* w, int64_t N, int64_t K, double* y) {
  for (int64_t n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) acc += a[k] * w[n * K + k];
    y[n] = acc;
  }
}

int64_t row_index(const int64_t* rows, int64_t i) { return rows ? rows[i] : i; }

}  // namespace

extern "C" {

int lo_version() { return 1; }

// bf16 bit patterns -> double, exactly.
void lo_widen(const uint16_t* bits, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = widen_one(bits[i]);
}

// Kept index pair (i0 < i1) of every group of four consecutive channels of every row of x (M x K doubles).
int lo_select_2of4(const double* x, int64_t M, int64_t K, int32_t* i0, int32_t* i1, int threads) {
  if (K % 4 != 0 || M < 0) return -2;
  parallel_rows(M, threads, [&](int64_t m) {
    for (int64_t g = 0; g < K / 4; ++g) {
      int a, b;
      select_group(x + m * K + 4 * g, &a, &b);
      i0[m * (K / 4) + g] = a;
      i1[m * (K / 4) + g] = b;
    }
  });
  return 0;
}

// keep (M x K bytes): 1 at the kept positions of every group.
int lo_keep_mask(const double* x, int64_t M, int64_t K, uint8_t* keep, int threads) {
  if (K % 4 != 0 || M < 0) return -2;
  parallel_rows(M, threads, [&](int64_t m) { keep_row(x + m * K, K, keep + m * K); });
  return 0;
}

// Per-row s of x (M x K doubles) given the kept positions.
int lo_norm_scale(const double* x, const uint8_t* keep, int64_t M, int64_t K, double* s, int threads) {
  if (M < 0 || K < 0) return -2;
  parallel_rows(M, threads, [&](int64_t m) { s[m] = scale_row(x + m * K, keep + m * K, K); });
  return 0;
}

// Canonical metadata bytes (M x G/2) of the kept pairs (M x G groups): nibble = i0 | i1 << 2, group 2j in the
// low nibble of byte j, group 2j + 1 in the high nibble.
int lo_canonical_meta(const int32_t* i0, const int32_t* i1, int64_t M, int64_t G, uint8_t* meta) {
  if (G % 2 != 0 || M < 0) return -2;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t j = 0; j < G / 2; ++j) {
      const int64_t a = m * G + 2 * j, b = a + 1;
      const uint32_t lo = static_cast<uint32_t>(i0[a] | (i1[a] << 2));
      const uint32_t hi = static_cast<uint32_t>(i0[b] | (i1[b] << 2));
      meta[m * (G / 2) + j] = static_cast<uint8_t>(lo | (hi << 4));
    }
  }
  return 0;
}

// S(X) in compressed form (what the sparsification step hands to the sparse GEMM):
//   keep  M x K bytes, 1 at the kept positions;
//   vals  M x K/2 bf16 bit patterns, the two kept entries of each group, lower position first;
//   meta  M x K/8 canonical bytes (may be NULL; requires K % 8 == 0 otherwise);
//   s     M doubles.
int lo_sparsify(const uint16_t* X, int64_t M, int64_t K, uint8_t* keep, uint16_t* vals, uint8_t* meta, double* s,
                int threads) {
  if (K % 4 != 0 || M < 0 || (meta && K % 8 != 0)) return -2;
  parallel_rows(M, threads, [&](int64_t m) {
    std::vector<double> x(static_cast<size_t>(K));
    for (int64_t k = 0; k < K; ++k) x[static_cast<size_t>(k)] = widen_one(X[m * K + k]);
    uint8_t* kp = keep + m * K;
    keep_row(x.data(), K, kp);
    s[m] = scale_row(x.data(), kp, K);
    int64_t v = 0;
    for (int64_t k = 0; k < K; ++k)
      if (kp[k]) vals[m * (K / 2) + v++] = X[m * K + k];
    if (meta) {
      for (int64_t j = 0; j < K / 8; ++j) {
        uint32_t byte = 0;
        for (int h = 0; h < 2; ++h) {
          const uint8_t* gk = kp + 8 * j + 4 * h;
          int first = -1, second = -1;
          for (int p = 0; p < 4; ++p)
            if (gk[p]) (first < 0 ? first : second) = p;
          byte |= static_cast<uint32_t>(first | (second << 2)) << (4 * h);
        }
        meta[m * (K / 8) + j] = static_cast<uint8_t>(byte);
      }
    }
  });
  return 0;
}

// Y = S(X) W^T + X (LA LB)^T in double: Y[i, :] for row rows[i] (all M rows in order when rows is NULL).
int lo_linear(const uint16_t* X, const uint16_t* W, const uint16_t* LA, const uint16_t* LB, int64_t M, int64_t N,
              int64_t K, int64_t R, const int64_t* rows, int64_t nrows, double* Y, int threads) {
  if (K % 4 != 0 || M < 0 || N < 0 || R < 0) return -2;
  const int64_t n_out = rows ? nrows : M;
  const std::vector<double> w = widen_all(W, N * K), la = widen_all(LA, N * R), lb = widen_all(LB, R * K);
  parallel_rows(n_out, threads, [&](int64_t i) {
    const int64_t m = row_index(rows, i);
    std::vector<double> x(static_cast<size_t>(K)), xt(static_cast<size_t>(K)), ys(static_cast<size_t>(N)),
        yr(static_cast<size_t>(N));
    std::vector<uint8_t> keep(static_cast<size_t>(K));
    for (int64_t k = 0; k < K; ++k) x[static_cast<size_t>(k)] = widen_one(X[m * K + k]);
    keep_row(x.data(), K, keep.data());
    const double s = scale_row(x.data(), keep.data(), K);
    for (int64_t k = 0; k < K; ++k) xt[static_cast<size_t>(k)] = keep[static_cast<size_t>(k)] ? x[static_cast<size_t>(k)] : 0.0;
    product_row(xt.data(), w.data(), N, K, ys.data());    // X~ W^T
    lora_row(x.data(), la.data(), lb.data(), N, K, R, yr.data());  // (X LB^T) LA^T
    for (int64_t n = 0; n < N; ++n) Y[i * N + n] = s * ys[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];
  });
  return 0;
}

// First factor of the LoRA branch, T[m, r] = sum_k X[m,k] LB[r,k], divided by s[m] when s is not NULL (the
// division lets the sparse branch and the LoRA branch share one accumulator scaled by s at the end).
int lo_lora_down(const uint16_t* X, const uint16_t* LB, const double* s, int64_t M, int64_t K, int64_t R, double* T,
                 int threads) {
  if (M < 0 || K < 0 || R < 0) return -2;
  const std::vector<double> lb = widen_all(LB, R * K);
  parallel_rows(M, threads, [&](int64_t m) {
    for (int64_t r = 0; r < R; ++r) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += widen_one(X[m * K + k]) * lb[static_cast<size_t>(r * K + k)];
      T[m * R + r] = s ? acc / s[m] : acc;
    }
  });
  return 0;
}

// A selectively skipped layer: Y = X W^T (+ X (LA LB)^T when LA and LB are both given).
int lo_linear_dense(const uint16_t* X, const uint16_t* W, const uint16_t* LA, const uint16_t* LB, int64_t M,
                    int64_t N, int64_t K, int64_t R, const int64_t* rows, int64_t nrows, double* Y, int threads) {
  if (M < 0 || N < 0 || K < 0 || ((LA == nullptr) != (LB == nullptr))) return -2;
  const int64_t n_out = rows ? nrows : M;
  const std::vector<double> w = widen_all(W, N * K);
  const std::vector<double> la = LA ? widen_all(LA, N * R) : std::vector<double>();
  const std::vector<double> lb = LB ? widen_all(LB, R * K) : std::vector<double>();
  parallel_rows(n_out, threads, [&](int64_t i) {
    const int64_t m = row_index(rows, i);
    std::vector<double> x(static_cast<size_t>(K)), y(static_cast<size_t>(N)), yr(static_cast<size_t>(N), 0.0);
    for (int64_t k = 0; k < K; ++k) x[static_cast<size_t>(k)] = widen_one(X[m * K + k]);
    product_row(x.data(), w.data(), N, K, y.data());
    if (LA) lora_row(x.data(), la.data(), lb.data(), N, K, R, yr.data());
    for (int64_t n = 0; n < N; ++n) Y[i * N + n] = y[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];
  });
  return 0;
}

// The weight-2:4 comparator: Y = X W~^T (+ X (LA LB)^T), W~ keeping the two largest |w| of every group of four
// consecutive input channels of each row of W (ties to the lower index), no rescaling.
int lo_linear_wsparse(const uint16_t* X, const uint16_t* W, const uint16_t* LA, const uint16_t* LB, int64_t M,
                      int64_t N, int64_t K, int64_t R, const int64_t* rows, int64_t nrows, double* Y, int threads) {
  if (K % 4 != 0 || M < 0 || N < 0 || ((LA == nullptr) != (LB == nullptr))) return -2;
  const int64_t n_out = rows ? nrows : M;
  std::vector<double> wt = widen_all(W, N * K);
  parallel_rows(N, threads, [&](int64_t n) {
    std::vector<uint8_t> keep(static_cast<size_t>(K));
    keep_row(wt.data() + n * K, K, keep.data());
    for (int64_t k = 0; k < K; ++k)
      if (!keep[static_cast<size_t>(k)]) wt[static_cast<size_t>(n * K + k)] = 0.0;
  });
  const std::vector<double> la = LA ? widen_all(LA, N * R) : std::vector<double>();
  const std::vector<double> lb = LB ? widen_all(LB, R * K) : std::vector<double>();
  parallel_rows(n_out, threads, [&](int64_t i) {
    const int64_t m = row_index(rows, i);
    std::vector<double> x(static_cast<size_t>(K)), y(static_cast<size_t>(N)), yr(static_cast<size_t>(N), 0.0);
    for (int64_t k = 0; k < K; ++k) x[static_cast<size_t>(k)] = widen_one(X[m * K + k]);
    product_row(x.data(), wt.data(), N, K, y.data());
    if (LA) lora_row(x.data(), la.data(), lb.data(), N, K, R, yr.data());
    for (int64_t n = 0; n < N; ++n) Y[i * N + n] = y[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];
  });
  return 0;
}

// Round to the nearest bf16 value, ties to even (8 significant bits), returned as its bit pattern.  Values too
// large for bf16 become infinity; NaN becomes the canonical quiet NaN.
uint16_t lo_round_bf16_one(double v) {
  if (std::isnan(v)) return 0x7FC0;
  const bool neg = std::signbit(v);
  const double a = std::fabs(v);
  float f = 0.0f;
  if (a != 0.0) {
    int e = 0;
    const double m = std::frexp(a, &e);              // a = m 2^e, m in [0.5, 1)
    int emin = -125;                                 // bf16 shares float32's exponent range
    double r;
    if (e >= emin) {
      r = std::nearbyint(std::ldexp(m, 8));          // 8 significant bits, ties to even
      f = static_cast<float>(std::ldexp(r, e - 8));  // exact: r has at most 9 bits
    } else {                                         // subnormal: a fixed quantum of 2^-133
      r = std::nearbyint(std::ldexp(a, 133));
      f = static_cast<float>(std::ldexp(r, -133));
    }
    if (std::isinf(f) || std::fabs(static_cast<double>(f)) > 3.3895313892515355e38) f = INFINITY;
  }
  if (neg) f = -f;
  uint32_t u;
  std::memcpy(&u, &f, sizeof(u));
  return static_cast<uint16_t>(u >> 16);
}

void lo_round_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = lo_round_bf16_one(x[i]);
}

// GELU with the exact error function: 0.5 x (1 + erf(x / sqrt(2))).
void lo_gelu(const double* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = 0.5 * x[i] * (1.0 + std::erf(x[i] / std::sqrt(2.0)));
}

// The MLP activation applied to a bf16 tensor (the up layer's bf16 output): H = bf16(GELU(Y)).
void lo_gelu_bf16(const uint16_t* Y, int64_t n, uint16_t* H) {
  for (int64_t i = 0; i < n; ++i) {
    const double y = widen_one(Y[i]);
    H[i] = lo_round_bf16_one(0.5 * y * (1.0 + std::erf(y / std::sqrt(2.0))));
  }
}

}  // extern "C"
