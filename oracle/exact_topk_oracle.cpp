// CPU oracle for exact row-wise FP32 Top-K over ragged rows.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file: only tests/, __graft_entry__.smoke() and bench.py's
// cpu_baseline / reference legs use it.  It shares no code, header, table or
// constant generator with the CUDA library.
//
// Two independent things live here, both written for a reader to check
// against the paper "Sample-Guided Exact Top-K Selection for Long-Context
// Sparse Attention" by eye:
//
//  1. oracle_topk_rows: the plain definition of the operator (section 2.1,
//     "Operator contract"; exactness criterion eq. 30 in section 6.1).  Each
//     row keeps the K largest valid scores, found with std::nth_element on
//     the total-order key of the FP32 bit pattern.  Rows with L <= K return
//     every valid index followed by -1.
//
//  2. oracle_method_trace: the three-phase method itself, step by step in the
//     paper's order and notation (sections 4.2-4.4, eqs. 11-25), with
//     straightforward loops.  It reports, per row, the route taken (Table 2 of
//     section 4.6), the Phase-1 boundaries tau0 / tau1, the admitted counts
//     C(tau), the exact coarse boundary tau*, |E0| and |Q0|, and produces its
//     own Top-K through the prefix-commit-retain recurrence.  The tests pin it
//     to the definition above and to brute force, and the GPU path must match
//     its per-row trace exactly.
//
// Floating point: no float arithmetic is used; every decision is taken on
// integer keys derived from the IEEE-754 bit patterns, so results do not
// depend on FTZ or rounding modes.  The FP16 projection (section 4.2,
// "round-to-nearest FP16 projection") is written out below from the IEEE-754
// binary16 definition.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Keys (section 4.2 eq. 11 and section 4.3 "descending sortable key").
// ---------------------------------------------------------------------------

// Ascending total-order key of an FP32 bit pattern: flipping the sign bit of
// non-negative values and all bits of negative values makes unsigned integer
// order equal numeric order (with -0 just below +0).
inline uint32_t asc32_bits(uint32_t u) {
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Descending key kappa_down32: a larger score gets a smaller key.
inline uint32_t desc32_bits(uint32_t u) { return ~asc32_bits(u); }

inline uint32_t bits_of(float x) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  return u;
}

// Inverse of desc32_bits.
inline uint32_t bits_from_desc32(uint32_t k) {
  uint32_t a = ~k;  // ascending key
  return (a & 0x80000000u) ? (a & 0x7FFFFFFFu) : ~a;
}

// IEEE-754 binary32 -> binary16, round to nearest, ties to even.
// The value of a finite normal float is sig * 2^(E-23) with sig in
// [2^23, 2^24).  The binary16 grid spacing ("ulp") at that magnitude is
// 2^(E-10) for normal halves (E >= -14) and 2^-24 for subnormal halves.  We
// divide by the ulp with an explicit remainder and round the quotient.
uint16_t f16_rne_bits(uint32_t u) {
  const uint32_t sign = (u >> 16) & 0x8000u;
  const uint32_t exp = (u >> 23) & 0xFFu;
  const uint32_t man = u & 0x7FFFFFu;
  if (exp == 0xFFu) {  // infinity or NaN (NaN is outside the contract)
    if (man == 0) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | 0x7C00u | 0x200u | (man >> 13));
  }
  if (exp == 0) return (uint16_t)sign;  // zero or binary32 subnormal (< 2^-126): rounds to +-0
  const int E = (int)exp - 127;
  const uint32_t sig = man | 0x800000u;
  if (E < -25) return (uint16_t)sign;  // below half the smallest half subnormal
  const int ulpexp = (E >= -14) ? (E - 10) : -24;
  const int shift = ulpexp - (E - 23);  // 13 for normal halves, 14..24 for subnormal halves
  uint32_t q = sig >> shift;
  const uint32_t rem = sig & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1;
  if (E >= -14) {
    int biased = E + 15;
    if (q == 2048u) {  // rounding carried into the next binade
      q = 1024u;
      biased += 1;
    }
    if (biased >= 31) return (uint16_t)(sign | 0x7C00u);  // overflow to infinity
    return (uint16_t)(sign | ((uint32_t)biased << 10) | (q - 1024u));
  }
  // Subnormal half: q in [0, 1024]; q == 1024 is exactly the smallest normal.
  return (uint16_t)(sign | q);
}

// Coarse map c(x) = floor(kappa_down16(fp16(x)) / 2^5)  (eq. 11), B_c = 2048.
inline int coarse_bin_bits(uint32_t u) {
  const uint32_t h = f16_rne_bits(u);
  const uint32_t asc16 = (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  const uint32_t desc16 = (~asc16) & 0xFFFFu;
  return (int)(desc16 >> 5);
}

// Digit j of the 11+11+10 split of kappa_down32, most significant first
// (section 4.3, "D = 3 digits of widths 11 + 11 + 10").
inline uint32_t digit_of(uint32_t desc_key, int j) {
  if (j == 0) return desc_key >> 21;
  if (j == 1) return (desc_key >> 10) & 0x7FFu;
  return desc_key & 0x3FFu;
}

inline int digit_bins(int j) { return j == 2 ? 1024 : 2048; }

constexpr uint32_t kDescPosInf = 0x007FFFFFu;  // desc32 key of +inf
constexpr uint32_t kDescNegInf = 0xFF800000u;  // desc32 key of -inf

// Largest desc32 key T in the non-NaN range whose coarse bin is <= tau: the
// inclusive FP32 endpoint of the admitted prefix c(x) <= tau (section 4.3,
// "Its cutoff is the smallest FP32 value admitted by that prefix").  Because
// c is monotone along desc32 keys, a plain binary search finds it.  Returns
// kDescPosInf - 1 (nothing admitted) when tau is below c(+inf).
uint32_t cutoff_for_bin(int tau) {
  if (coarse_bin_bits(bits_from_desc32(kDescPosInf)) > tau) return kDescPosInf - 1;
  uint32_t lo = kDescPosInf, hi = kDescNegInf;  // invariant: c(lo) <= tau
  while (lo < hi) {
    const uint32_t mid = lo + (uint32_t)(((uint64_t)(hi - lo) + 1) / 2);
    if (coarse_bin_bits(bits_from_desc32(mid)) <= tau)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

inline int64_t clamp_len(int64_t v, int64_t n) { return v < 0 ? 0 : (v > n ? n : v); }

// ---------------------------------------------------------------------------
// 1. The plain definition.
// ---------------------------------------------------------------------------

void topk_definition_row(const float* x, int64_t L, int K, int32_t* out) {
  if (L <= K) {
    for (int64_t i = 0; i < L; ++i) out[i] = (int32_t)i;
    for (int64_t i = L; i < K; ++i) out[i] = -1;
    return;
  }
  std::vector<std::pair<uint32_t, int32_t>> items((size_t)L);
  for (int64_t i = 0; i < L; ++i) items[(size_t)i] = {asc32_bits(bits_of(x[i])), (int32_t)i};
  // Larger key first; among equal keys the smaller index first (any tie
  // choice is allowed by the contract; this one is simply deterministic).
  auto better = [](const std::pair<uint32_t, int32_t>& a, const std::pair<uint32_t, int32_t>& b) {
    return a.first != b.first ? a.first > b.first : a.second < b.second;
  };
  std::nth_element(items.begin(), items.begin() + (K - 1), items.end(), better);
  for (int k = 0; k < K; ++k) out[k] = items[(size_t)k].second;
}

template <class F>
void parallel_rows(int64_t rows, int nthreads, F fn) {
  if (nthreads <= 1 || rows <= 1) {
    for (int64_t r = 0; r < rows; ++r) fn(r);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t T = std::min<int64_t>(nthreads, rows);
  pool.reserve((size_t)T);
  for (int64_t t = 0; t < T; ++t)
    pool.emplace_back([&, t]() {
      for (int64_t r = t; r < rows; r += T) fn(r);
    });
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------------------
// 2. The three-phase method, written out (sections 4.2-4.4).
// ---------------------------------------------------------------------------

// Route codes.  Table 2 of section 4.6 lists the five routes of a row with
// L > K; the pad route covers L <= K (section 2.1), and the guess routes
// cover an optional previous-step Top-K used as the proposal.
enum Route {
  kRoutePad = 0,
  kRoutePrimary = 1,
  kRouteBand = 2,
  kRouteExactAfterBand = 3,
  kRouteExactNoBand = 4,
  kRouteDirectExact = 5,
  kRouteGuess = 6,
  kRouteGuessExact = 7,
};

// Per-row trace fields, in order.
enum TraceField {
  kTrRoute = 0,
  kTrTau0 = 1,     // primary boundary tau0 (or the guessed boundary)
  kTrTau1 = 2,     // secondary boundary tau1
  kTrC0 = 3,       // C(tau0)
  kTrC1 = 4,       // C(tau1) when the band was attempted
  kTrTauStar = 5,  // exact coarse boundary tau*
  kTrE0 = 6,       // |E0|
  kTrQ0 = 7,       // |Q0|
  kTrFields = 8,
};

struct MethodParams {
  int K;
  int s;          // view stride (power of two)
  int dual;       // 1: record tau1 and attempt the band on underfill
  int rho0_num, rho0_den;  // K~ = rho0 * K
  int rho1_num, rho1_den;  // K~1 = rho1 * K
  int sampled;    // 0: every row with L > K takes the direct-exact route
};

// pi_s: bit reversal of the log2(s) low bits (the pages only ask for "a fixed
// permutation of the s residue classes").
int view_phase(int64_t r, int s) {
  int bits = 0;
  while ((1 << bits) < s) ++bits;
  const int v = (int)(r % s);
  int out = 0;
  for (int b = 0; b < bits; ++b)
    if (v & (1 << b)) out |= 1 << (bits - 1 - b);
  return out;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Phase 3 (eqs. 22-25) over frontier Q with remaining quota k; appends the
// committed indices to out_sel.  Keys are kappa_down32.
void phase3_refine(const float* x, std::vector<int32_t> Q, int64_t k, std::vector<int32_t>& out_sel) {
  for (int j = 0; j < 3 && k > 0; ++j) {
    const int B = digit_bins(j);
    std::vector<int64_t> h((size_t)B, 0);
    for (int32_t i : Q) h[digit_of(desc32_bits(bits_of(x[i])), j)] += 1;
    // b_j = min{b : H_j(b) >= k_j}  (eq. 23)
    int64_t H = 0;
    int bj = -1;
    for (int b = 0; b < B; ++b) {
      H += h[(size_t)b];
      if (H >= k) {
        bj = b;
        break;
      }
    }
    std::vector<int32_t> next;
    int64_t committed = 0;
    for (int32_t i : Q) {
      const uint32_t d = digit_of(desc32_bits(bits_of(x[i])), j);
      if ((int)d < bj) {  // R_j (eq. 24)
        out_sel.push_back(i);
        ++committed;
      } else if ((int)d == bj) {  // Q_{j+1} (eq. 25)
        next.push_back(i);
      }
    }
    k -= committed;
    Q.swap(next);
  }
  // After the last digit every key in Q is identical; fill the rest from it.
  for (int64_t t = 0; t < k; ++t) out_sel.push_back(Q[(size_t)t]);
}

void method_row(const float* x, int64_t L, int64_t r, const MethodParams& p, const int32_t* guess,
                int32_t* out, int32_t* tr) {
  const int K = p.K;
  for (int f = 0; f < kTrFields; ++f) tr[f] = -1;
  if (L <= K) {
    tr[kTrRoute] = kRoutePad;
    for (int64_t i = 0; i < L; ++i) out[i] = (int32_t)i;
    for (int64_t i = L; i < K; ++i) out[i] = -1;
    return;
  }
  std::vector<int> c((size_t)L);
  for (int64_t i = 0; i < L; ++i) c[(size_t)i] = coarse_bin_bits(bits_of(x[i]));
  auto admitted_count = [&](int tau) {
    int64_t n = 0;
    for (int64_t i = 0; i < L; ++i) n += c[(size_t)i] <= tau;
    return n;
  };
  std::vector<int32_t> sel;
  sel.reserve((size_t)K);
  int route = -1;
  int tau_used = -1;

  // Optional guess source: the previous step's K indices.  Used only when all
  // K entries are valid positions of this row.
  bool guess_ok = false;
  if (guess) {
    guess_ok = true;
    int worst = -1;
    for (int t = 0; t < K; ++t) {
      const int32_t g = guess[t];
      if (g < 0 || g >= L) {
        guess_ok = false;
        break;
      }
      worst = std::max(worst, c[(size_t)g]);
    }
    if (guess_ok) {
      tr[kTrTau0] = worst;
      const int64_t C0 = admitted_count(worst);
      tr[kTrC0] = (int32_t)C0;
      if (C0 >= K) {
        route = kRouteGuess;
        tau_used = worst;
      } else {
        route = kRouteGuessExact;
      }
    }
  }

  if (!guess_ok) {
    bool usable = false;
    if (p.sampled) {
      // Phase 1 (section 4.2): the row-phased view V = {i < L : i = a_r mod s}
      // and its coarse histogram / inclusive prefix (eq. 14).
      const int a = view_phase(r, p.s);
      std::vector<int64_t> h(2048, 0);
      int64_t nv = 0;
      for (int64_t i = a; i < L; i += p.s) {
        h[(size_t)c[(size_t)i]] += 1;
        ++nv;
      }
      const int64_t q0 = ceil_div((int64_t)p.rho0_num * K, (int64_t)p.rho0_den * p.s);
      const int64_t q1 = ceil_div((int64_t)p.rho1_num * K, (int64_t)p.rho1_den * p.s);
      const int64_t qmax = p.dual ? q1 : q0;
      usable = nv >= qmax;  // section 5.2, "A view is usable only when..."
      if (usable) {
        int tau0 = -1, tau1 = -1;
        int64_t H = 0;
        for (int b = 0; b < 2048; ++b) {
          H += h[(size_t)b];
          if (tau0 < 0 && H >= q0) tau0 = b;  // eq. 15
          if (tau1 < 0 && H >= q1) tau1 = b;
        }
        tr[kTrTau0] = tau0;
        if (p.dual) tr[kTrTau1] = tau1;
        // Phase 2 (section 4.3): admitted tail and its certificate.
        const int64_t C0 = admitted_count(tau0);
        tr[kTrC0] = (int32_t)C0;
        if (C0 >= K) {
          route = kRoutePrimary;
          tau_used = tau0;
        } else if (p.dual) {
          const int64_t C1 = admitted_count(tau1);  // band rescue, eqs. 18-19
          tr[kTrC1] = (int32_t)C1;
          if (C1 >= K) {
            route = kRouteBand;
            tau_used = tau1;
          } else {
            route = kRouteExactAfterBand;
          }
        } else {
          route = kRouteExactNoBand;
        }
      }
    }
    if (!usable) route = kRouteDirectExact;
  }

  std::vector<int32_t> Q0;
  int64_t k0 = K;
  if (tau_used >= 0) {
    // Certified sampled route: E0 = {}, Q0 = A(tau), k0 = K  (eq. 21).
    for (int64_t i = 0; i < L; ++i)
      if (c[(size_t)i] <= tau_used) Q0.push_back((int32_t)i);
    tr[kTrE0] = 0;
  } else {
    // Exact coarse recovery (eq. 20): tau* = min{b : C(b) >= K}.
    std::vector<int64_t> h(2048, 0);
    for (int64_t i = 0; i < L; ++i) h[(size_t)c[(size_t)i]] += 1;
    int64_t H = 0;
    int tau_star = -1;
    for (int b = 0; b < 2048; ++b) {
      if (H + h[(size_t)b] >= K) {
        tau_star = b;
        break;
      }
      H += h[(size_t)b];
    }
    tr[kTrTauStar] = tau_star;
    for (int64_t i = 0; i < L; ++i) {
      if (c[(size_t)i] < tau_star)
        sel.push_back((int32_t)i);  // E0
      else if (c[(size_t)i] == tau_star)
        Q0.push_back((int32_t)i);
    }
    tr[kTrE0] = (int32_t)sel.size();
    k0 = K - (int64_t)sel.size();
  }
  tr[kTrQ0] = (int32_t)Q0.size();
  tr[kTrRoute] = route;
  phase3_refine(x, std::move(Q0), k0, sel);
  for (int k = 0; k < K; ++k) out[k] = sel[(size_t)k];
}

}  // namespace

extern "C" {

// Plain definition of the operator for rows [0, M_live) of an [M, pitch]
// float32 matrix; rows >= M_live of `out` are left untouched.
int oracle_topk_rows(const float* X, int64_t M, int64_t N, int64_t pitch, const int32_t* ke,
                     int64_t M_live, int K, int32_t* out, int nthreads) {
  if (!X || !ke || !out || K < 1 || N < 0 || pitch < N || M < 0) return -1;
  if (M_live > M) M_live = M;
  parallel_rows(M_live, nthreads, [&](int64_t r) {
    topk_definition_row(X + r * pitch, clamp_len(ke[r], N), K, out + r * (int64_t)K);
  });
  return 0;
}

// The three-phase method with its per-row trace (kTrFields int32 per row).
// `guess` is an optional [M, K] int32 array of previous-step indices.
int oracle_method_trace(const float* X, int64_t M, int64_t N, int64_t pitch, const int32_t* ke,
                        int64_t M_live, int K, int s, int dual, int rho0_num, int rho0_den,
                        int rho1_num, int rho1_den, int sampled, const int32_t* guess,
                        int32_t* out, int32_t* trace, int nthreads) {
  if (!X || !ke || !out || !trace || K < 1 || N < 0 || pitch < N || M < 0) return -1;
  if (s < 1 || (s & (s - 1)) != 0) return -2;
  if (M_live > M) M_live = M;
  const MethodParams p{K, s, dual, rho0_num, rho0_den, rho1_num, rho1_den, sampled};
  parallel_rows(M_live, nthreads, [&](int64_t r) {
    method_row(X + r * pitch, clamp_len(ke[r], N), r, p, guess ? guess + r * (int64_t)K : nullptr,
               out + r * (int64_t)K, trace + r * (int64_t)kTrFields);
  });
  return 0;
}

// Scalar helpers, exported so the tests can pin each against independent
// definitions (numpy's binary16 cast, hand-computed values, monotonicity).
uint16_t oracle_f16_bits(float x) { return f16_rne_bits(bits_of(x)); }
int oracle_coarse_bin(float x) { return coarse_bin_bits(bits_of(x)); }
uint32_t oracle_desc32(float x) { return desc32_bits(bits_of(x)); }
uint32_t oracle_cutoff_for_bin(int tau) { return cutoff_for_bin(tau); }
int oracle_view_phase(int64_t r, int s) { return view_phase(r, s); }

void oracle_f16_bits_array(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f16_rne_bits(bits_of(x[i]));
}
void oracle_coarse_bin_array(const float* x, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = coarse_bin_bits(bits_of(x[i]));
}

int oracle_hardware_threads(void) {
  const unsigned n = std::thread::hardware_concurrency();
  return n ? (int)n : 1;
}

}  // extern "C"
