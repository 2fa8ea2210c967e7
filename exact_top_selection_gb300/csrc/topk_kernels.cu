// Exact row-wise FP32 Top-K kernels for sm_103a.
//
// Implements the sample-guided three-phase selector of "Sample-Guided Exact
// Top-K Selection for Long-Context Sparse Attention" (sections 4.2-4.5) as
// three kernel families behind one launcher (section 5.5):
//
//   persistent_sampled_kernel  one 512-thread CTA owns a row for all phases;
//                              rows after the first wave come from a device
//                              queue in completion order.
//   kv_split_kernel            P CTAs scan disjoint segments of one row and
//                              publish their candidate ranges; the last CTA to
//                              arrive merges them (eq. 27) and finishes the row.
//   row_local_exact_kernel     one 1024-thread CTA per row takes the exact
//                              coarse route directly; short rows stay in
//                              registers between the two classification passes.
//
// Every route ends in the same refinement interface (E0, Q0, k0, h0) of eqs.
// 20-21 and the 11+11+10 prefix-commit-retain recurrence of eqs. 22-25.
//
// Keys.  kappa_down32 (section 4.3) is computed from the FP32 bit pattern u as
// u for negative scores and u ^ 0x7FFFFFFF otherwise, so that a larger score has
// a smaller unsigned key and -0 ranks just below +0.  The coarse bin c(x) of eq.
// 11 is the top 11 bits of the same transform of the round-to-nearest FP16
// projection.  NaN is outside the contract; to keep c monotone along the full
// key space (and so every count consistent) positive NaNs are placed in bin 0
// and negative NaNs in bin 2047, matching their key order.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "etk_internal.h"

namespace etk {
namespace {

constexpr int kCoarseBins = 2048;
constexpr uint32_t kDescPosInf = 0x007FFFFFu;  // kappa_down32(+inf)
constexpr uint32_t kDescNegInf = 0xFF800000u;  // kappa_down32(-inf)
constexpr unsigned kFull = 0xFFFFFFFFu;

// ----------------------------------------------------------------------------
// Keys and the coarse map
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t desc_key(uint32_t u) {
  return u ^ (~(uint32_t)((int32_t)u >> 31) & 0x7FFFFFFFu);
}

__device__ __forceinline__ uint32_t bits_from_desc(uint32_t d) {
  return (d & 0x80000000u) ? d : (d ^ 0x7FFFFFFFu);
}

// c(x) of eq. 11 given x's bit pattern u and its kappa_down32 key d.
__device__ __forceinline__ int coarse_bin(uint32_t u, uint32_t d) {
  if (d < kDescPosInf) return 0;
  if (d > kDescNegInf) return kCoarseBins - 1;
  const uint32_t h = __half_as_ushort(__float2half_rn(__uint_as_float(u)));
  const uint32_t d16 = (h & 0x8000u) ? h : (h ^ 0x7FFFu);
  return (int)(d16 >> 5);
}

// Largest kappa_down32 key whose coarse bin is <= tau: the inclusive FP32
// endpoint of the admitted prefix (section 4.3; section 5.2 "converts the
// selected bins to their inclusive FP32 endpoints").  c is non-decreasing along
// the key space, so a binary search finds it.
__device__ uint32_t cutoff_for_bin(int tau) {
  uint32_t lo = 0u, hi = 0xFFFFFFFFu;  // c(key 0) = 0 <= tau for tau >= 0
  while (lo < hi) {
    const uint32_t mid = lo + (uint32_t)((((uint64_t)(hi - lo)) + 1ull) >> 1);
    const uint32_t u = bits_from_desc(mid);
    if (coarse_bin(u, mid) <= tau)
      lo = mid;
    else
      hi = mid - 1u;
  }
  return lo;
}

// Digit j of the 11+11+10 split, most significant first (section 4.3).
__device__ __forceinline__ uint32_t digit(uint32_t d, int j) {
  return j == 0 ? (d >> 21) : (j == 1 ? ((d >> 10) & 0x7FFu) : (d & 0x3FFu));
}

// ----------------------------------------------------------------------------
// Loads
// ----------------------------------------------------------------------------

// Streaming 128-bit load of score bits that are read once per pass.
__device__ __forceinline__ uint4 ld_stream4(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream1(const float* p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ----------------------------------------------------------------------------
// Per-CTA shared state
// ----------------------------------------------------------------------------

struct alignas(16) RowState {
  uint32_t hist[kCoarseBins];  // one allocation: h_{r,s} -> h0 -> h1 -> h2 (Fig. 5)
  uint32_t warp_sums[32];
  int32_t res_bin[2];
  uint32_t res_below[2];
  uint32_t res_cnt[2];
  uint32_t n_front;  // frontier entries
  uint32_t n_out;    // output slots used
  uint32_t n_keep;   // survivors during an in-place compaction
  uint32_t cut[2];   // kappa_down32 cutoffs
  int32_t gmax;      // guess source: worst coarse bin
  int32_t ginvalid;  // guess source: an entry outside [0, L)
  int32_t next_row;
  int32_t is_last;
  uint32_t seg_c0;   // KV-split: this segment's primary candidates
  uint32_t seg_cb;   // KV-split: this segment's band candidates
  uint32_t total;    // KV-split finisher: merged count
  int32_t pad_[1];
};

struct Params {
  const float* logits;
  int64_t pitch;
  int32_t N;
  int32_t M_cap;
  int32_t K;
  int32_t s;
  int32_t s_bits;
  int32_t dual;
  int32_t q0;
  int32_t q1;
  int32_t P;
  int32_t cap;
  const int32_t* ke;
  int32_t* out;
  const int32_t* num_valid_rows;
  int32_t* counters;
  int32_t* ws_idx;   // [slices][N]
  uint32_t* ws_key;  // [slices][N]
  int32_t* seg_counts;  // [M_cap][P][2]
  const int32_t* prev;
  int32_t* trace;
};

// Candidate frontier: logical entries [0, cap) live in shared memory, entries
// at logical positions >= cap live at the same position of a global slice of
// capacity gcap (section 5.4: "Two global ping-pong slices extend the shared
// frontier"; here one slice suffices because compaction is done in place).
struct Frontier {
  int32_t* s_idx;
  uint32_t* s_key;
  uint32_t cap;
  int32_t* g_idx;
  uint32_t* g_key;
  uint32_t gcap;

  __device__ __forceinline__ void put(uint32_t p, int32_t i, uint32_t d) const {
    if (p < cap) {
      s_idx[p] = i;
      s_key[p] = d;
    } else if (p < gcap) {
      g_idx[p] = i;
      g_key[p] = d;
    }
  }
  __device__ __forceinline__ void get(uint32_t p, int32_t& i, uint32_t& d) const {
    if (p < cap) {
      i = s_idx[p];
      d = s_key[p];
    } else if (p < gcap) {
      i = __ldcg(g_idx + p);
      d = __ldcg(g_key + p);
    } else {
      i = -1;
      d = 0xFFFFFFFFu;
    }
  }
};

__device__ __forceinline__ void flag_status(int32_t* counters, int bit) {
  atomicOr(counters + kCtrStatus, bit);
}

template <int THREADS>
__device__ __forceinline__ void clear_hist(RowState& st, int nbins) {
  for (int b = threadIdx.x; b < nbins; b += THREADS) st.hist[b] = 0u;
}

// For each target t of `targets` (ntargets <= 2): res_bin = min{b : H(b) >= t}
// over the inclusive prefix H of hist[0, nbins), res_below = H(b - 1) and
// res_cnt = hist[b]; res_bin = -1 when the total is below t.  The histogram is
// only read.  Must be entered by the whole CTA after the histogram is complete;
// results are visible to every thread on return.
template <int THREADS>
__device__ void find_boundaries(RowState& st, int nbins, int ntargets, uint32_t t0, uint32_t t1) {
  constexpr int kWarps = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins / THREADS;  // nbins is 1024 or 2048, THREADS 512 or 1024
  const int b0 = tid * per;
  uint32_t local = 0;
  for (int k = 0; k < per; ++k) local += st.hist[b0 + k];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (tid < 2) {
    st.res_bin[tid] = -1;
    st.res_below[tid] = 0u;
    st.res_cnt[tid] = 0u;
  }
  if (lane == 31) st.warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? st.warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += v;
    }
    if (lane < kWarps) st.warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  uint32_t run = (warp ? st.warp_sums[warp - 1] : 0u) + (incl - local);
  for (int k = 0; k < per; ++k) {
    const uint32_t h = st.hist[b0 + k];
    const uint32_t prev = run;
    run += h;
    if (prev < t0 && t0 <= run) {
      st.res_bin[0] = b0 + k;
      st.res_below[0] = prev;
      st.res_cnt[0] = h;
    }
    if (ntargets > 1 && prev < t1 && t1 <= run) {
      st.res_bin[1] = b0 + k;
      st.res_below[1] = prev;
      st.res_cnt[1] = h;
    }
  }
  __syncthreads();
}

// ----------------------------------------------------------------------------
// Row scans
// ----------------------------------------------------------------------------

// Visits every valid element of row[lo, hi) once: 128-bit loads on the 16-byte
// aligned body, scalar loads on the unaligned head and the tail (section 5.3).
// fn(u, i) receives the FP32 bit pattern and the row index.
template <int THREADS, int UNROLL, class Fn>
__device__ __forceinline__ void for_each_in_range(const float* row, int lo, int hi, Fn&& fn) {
  if (lo >= hi) return;
  const int tid = threadIdx.x;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + lo);
  // Scores are 4-byte aligned (checked on the host): at most 3 head elements.
  int head = (int)(((16u - (uint32_t)(addr & 15u)) & 15u) >> 2);
  if (head > hi - lo) head = hi - lo;
  const int a0 = lo + head;
  const int nvec = (hi - a0) >> 2;
  const int a_end = a0 + (nvec << 2);
  if (tid < head) fn(ld_stream1(row + lo + tid), lo + tid);
  const uint4* v = reinterpret_cast<const uint4*>(row + a0);
  int j = tid;
  for (; j + (UNROLL - 1) * THREADS < nvec; j += UNROLL * THREADS) {
    uint4 x[UNROLL];
#pragma unroll
    for (int q = 0; q < UNROLL; ++q) x[q] = ld_stream4(v + j + q * THREADS);
#pragma unroll
    for (int q = 0; q < UNROLL; ++q) {
      const int i = a0 + ((j + q * THREADS) << 2);
      fn(x[q].x, i);
      fn(x[q].y, i + 1);
      fn(x[q].z, i + 2);
      fn(x[q].w, i + 3);
    }
  }
  for (; j < nvec; j += THREADS) {
    const uint4 x = ld_stream4(v + j);
    const int i = a0 + (j << 2);
    fn(x.x, i);
    fn(x.y, i + 1);
    fn(x.z, i + 2);
    fn(x.w, i + 3);
  }
  const int t = a_end + tid;
  if (t < hi) fn(ld_stream1(row + t), t);
}

// Output slot reservation for one committed index.
__device__ __forceinline__ void commit(RowState& st, int32_t* out_row, int K, int32_t i) {
  const uint32_t slot = atomicAdd(&st.n_out, 1u);
  if (slot < (uint32_t)K) out_row[slot] = i;
}

// Phase 2 (section 4.3, eq. 16-17; section 5.3): one pass over row[lo, hi)
// admits every index whose key d lies in [dlo, dlo + dspan], appends (i, d) to
// the frontier and adds digit 0 of d to the shared histogram.
template <int THREADS>
__device__ void scan_admit(const float* row, int lo, int hi, uint32_t dlo, uint32_t dspan,
                           const Frontier& F, RowState& st) {
  for_each_in_range<THREADS, 4>(row, lo, hi, [&](uint32_t u, int i) {
    const uint32_t d = desc_key(u);
    if (d - dlo <= dspan) {
      const uint32_t p = atomicAdd(&st.n_front, 1u);
      F.put(p, i, d);
      atomicAdd(&st.hist[d >> 21], 1u);
    }
  });
}

// Coarse histogram over row[lo, hi) (first pass of exact coarse recovery, eq. 20).
template <int THREADS>
__device__ void scan_coarse_hist(const float* row, int lo, int hi, RowState& st) {
  for_each_in_range<THREADS, 4>(row, lo, hi, [&](uint32_t u, int i) {
    atomicAdd(&st.hist[coarse_bin(u, desc_key(u))], 1u);
  });
}

// Second pass of exact coarse recovery (eq. 20): keys d <= tlo (c < tau*) are
// committed to the output (E0), keys in (tlo, thi] (c == tau*) form Q0 and h0.
template <int THREADS>
__device__ void scan_exact_classify(const float* row, int lo, int hi, bool has_lo, uint32_t tlo,
                                    uint32_t thi, const Frontier& F, RowState& st, int32_t* out_row,
                                    int K) {
  for_each_in_range<THREADS, 4>(row, lo, hi, [&](uint32_t u, int i) {
    const uint32_t d = desc_key(u);
    if (d <= thi) {
      if (has_lo && d <= tlo) {
        commit(st, out_row, K, i);
      } else {
        const uint32_t p = atomicAdd(&st.n_front, 1u);
        F.put(p, i, d);
        atomicAdd(&st.hist[d >> 21], 1u);
      }
    }
  });
}

// ----------------------------------------------------------------------------
// Phase 3: prefix-commit-retain refinement (section 4.4, eqs. 22-25)
// ----------------------------------------------------------------------------

// Entry: frontier holds n entries (Q0), st.hist holds h0 (digit 0 over Q0),
// k = k0 indices remain to be selected, st.n_out = |E0|.  Exit: st.n_out == K.
template <int THREADS>
__device__ void refine(const Frontier& F, uint32_t n, uint32_t k, RowState& st, int32_t* out_row,
                       int K) {
  constexpr int R = 4;
  constexpr uint32_t CH = THREADS * R;
  const int tid = threadIdx.x;
  for (int j = 0; j < 3 && k > 0; ++j) {
    const int nb = (j == 2) ? 1024 : 2048;
    find_boundaries<THREADS>(st, nb, 1, k, 0u);
    const int b = st.res_bin[0];
    const uint32_t below = st.res_below[0];
    const uint32_t cnt = st.res_cnt[0];
    if (b < 0) {  // inconsistent counts: cannot happen; finish_row flags it
      k = 0;
      break;
    }
    if (below + cnt == k) {
      // The boundary group completes the quota exactly: commit every entry
      // whose digit is <= b and stop.
      for (uint32_t p = tid; p < n; p += THREADS) {
        int32_t i;
        uint32_t d;
        F.get(p, i, d);
        if ((int)digit(d, j) <= b) commit(st, out_row, K, i);
      }
      k = 0;
      break;
    }
    __syncthreads();  // every thread has read res_* before hist is cleared
    const bool next = j < 2;
    if (next) clear_hist<THREADS>(st, 2048);
    if (tid == 0) st.n_keep = 0u;
    __syncthreads();
    if (below == 0u && cnt == n) {
      // Whole frontier in the boundary group: nothing to commit or move;
      // only the next digit's histogram is needed.
      if (next) {
        for (uint32_t p = tid; p < n; p += THREADS) {
          int32_t i;
          uint32_t d;
          F.get(p, i, d);
          atomicAdd(&st.hist[digit(d, j + 1)], 1u);
        }
      }
    } else {
      // In-place compaction in chunks: every entry of a chunk is read before
      // any survivor of that chunk is written, and survivors land at
      // positions below the chunk's end, so no unread entry is overwritten.
      for (uint32_t c0 = 0; c0 < n; c0 += CH) {
        int32_t idx[R];
        uint32_t key[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t p = c0 + r * THREADS + tid;
          if (p < n)
            F.get(p, idx[r], key[r]);
          else
            idx[r] = -2;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (idx[r] == -2) continue;
          const int dg = (int)digit(key[r], j);
          if (dg < b) {
            commit(st, out_row, K, idx[r]);
          } else if (dg == b) {
            const uint32_t q = atomicAdd(&st.n_keep, 1u);
            F.put(q, idx[r], key[r]);
            if (next) atomicAdd(&st.hist[digit(key[r], j + 1)], 1u);
          }
        }
        __syncthreads();
      }
      n = cnt;
      k -= below;
    }
    __syncthreads();
  }
  if (k > 0) {
    // After the last digit every remaining key is identical: fill from it.
    for (uint32_t p = tid; p < k && p < n; p += THREADS) {
      int32_t i;
      uint32_t d;
      F.get(p, i, d);
      commit(st, out_row, K, i);
    }
  }
  __syncthreads();
}

// ----------------------------------------------------------------------------
// Row-level building blocks
// ----------------------------------------------------------------------------

template <int THREADS>
__device__ void write_pad_row(int32_t* out_row, int L, int K) {
  for (int t = threadIdx.x; t < K; t += THREADS) out_row[t] = t < L ? t : -1;
}

__device__ __forceinline__ void write_trace(const Params& p, int row, int route, int tau0, int tau1,
                                            int c0, int c1, int tstar, int e0, int q0) {
  if (p.trace == nullptr || threadIdx.x != 0) return;
  int32_t* t = p.trace + (int64_t)row * EXACT_TOPK_TRACE_FIELDS;
  t[0] = route;
  t[1] = tau0;
  t[2] = tau1;
  t[3] = c0;
  t[4] = c1;
  t[5] = tstar;
  t[6] = e0;
  t[7] = q0;
}

// Final guard: every slot must be written exactly once.
template <int THREADS>
__device__ void finish_row(const Params& p, RowState& st, int32_t* out_row) {
  __syncthreads();
  const uint32_t used = st.n_out;
  if (used != (uint32_t)p.K) {
    for (uint32_t t = used + threadIdx.x; t < (uint32_t)p.K; t += THREADS) out_row[t] = -1;
    if (threadIdx.x == 0) flag_status(p.counters, 1);
  }
  __syncthreads();
}

// Exact coarse recovery over row[0, L) followed by refinement (eq. 20).
// Leaves st.n_out == K.  Returns tau*, |E0| and |Q0| through the out params.
template <int THREADS>
__device__ void exact_route(const Params& p, const float* row, int L, const Frontier& F, RowState& st,
                            int32_t* out_row, int& tstar, int& e0, int& q0n) {
  const int K = p.K;
  clear_hist<THREADS>(st, 2048);
  if (threadIdx.x == 0) {
    st.n_front = 0u;
    st.n_out = 0u;
  }
  __syncthreads();
  scan_coarse_hist<THREADS>(row, 0, L, st);
  __syncthreads();
  find_boundaries<THREADS>(st, 2048, 1, (uint32_t)K, 0u);
  tstar = st.res_bin[0];
  e0 = (int)st.res_below[0];
  if (threadIdx.x == 0) {
    st.cut[1] = cutoff_for_bin(tstar);
  } else if (threadIdx.x == 32) {
    st.cut[0] = tstar > 0 ? cutoff_for_bin(tstar - 1) : 0u;
  }
  __syncthreads();
  clear_hist<THREADS>(st, 2048);
  __syncthreads();
  scan_exact_classify<THREADS>(row, 0, L, tstar > 0, st.cut[0], st.cut[1], F, st, out_row, K);
  __syncthreads();
  q0n = (int)st.n_front;
  refine<THREADS>(F, st.n_front, (uint32_t)(K - e0), st, out_row, K);
}

// Row-local exact route with the row resident in registers (section 5.5,
// "Row-local exact": the short-row specialization keeps aligned score vectors
// in registers across boundary construction and classification).
template <int THREADS, int VPT>
__device__ void exact_route_resident(const Params& p, const float* row, int L, const Frontier& F,
                                     RowState& st, int32_t* out_row, int& tstar, int& e0, int& q0n) {
  const int K = p.K;
  const int tid = threadIdx.x;
  uint32_t v[VPT];
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15u) == 0u;
#pragma unroll
  for (int g = 0; g < VPT / 4; ++g) {
    const int i0 = (g * THREADS + tid) * 4;
    if (aligned && i0 + 3 < L) {
      const uint4 x = ld_stream4(reinterpret_cast<const uint4*>(row + i0));
      v[g * 4 + 0] = x.x;
      v[g * 4 + 1] = x.y;
      v[g * 4 + 2] = x.z;
      v[g * 4 + 3] = x.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[g * 4 + e] = (i0 + e < L) ? ld_stream1(row + i0 + e) : 0u;
    }
  }
  clear_hist<THREADS>(st, 2048);
  if (tid == 0) {
    st.n_front = 0u;
    st.n_out = 0u;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < VPT / 4; ++g) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = (g * THREADS + tid) * 4 + e;
      if (i < L) atomicAdd(&st.hist[coarse_bin(v[g * 4 + e], desc_key(v[g * 4 + e]))], 1u);
    }
  }
  __syncthreads();
  find_boundaries<THREADS>(st, 2048, 1, (uint32_t)K, 0u);
  tstar = st.res_bin[0];
  e0 = (int)st.res_below[0];
  if (tid == 0) {
    st.cut[1] = cutoff_for_bin(tstar);
  } else if (tid == 32) {
    st.cut[0] = tstar > 0 ? cutoff_for_bin(tstar - 1) : 0u;
  }
  __syncthreads();
  clear_hist<THREADS>(st, 2048);
  __syncthreads();
  const uint32_t tlo = st.cut[0], thi = st.cut[1];
  const bool has_lo = tstar > 0;
#pragma unroll
  for (int g = 0; g < VPT / 4; ++g) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = (g * THREADS + tid) * 4 + e;
      if (i < L) {
        const uint32_t d = desc_key(v[g * 4 + e]);
        if (d <= thi) {
          if (has_lo && d <= tlo) {
            commit(st, out_row, K, i);
          } else {
            const uint32_t q = atomicAdd(&st.n_front, 1u);
            F.put(q, i, d);
            atomicAdd(&st.hist[d >> 21], 1u);
          }
        }
      }
    }
  }
  __syncthreads();
  q0n = (int)st.n_front;
  refine<THREADS>(F, st.n_front, (uint32_t)(K - e0), st, out_row, K);
}

__device__ __forceinline__ int view_phase(int row, int s, int s_bits) {
  if (s_bits == 0) return 0;
  return (int)(__brev((uint32_t)(row & (s - 1))) >> (32 - s_bits));
}

__device__ __forceinline__ int view_size(int L, int a, int s) {
  return L > a ? (L - a + s - 1) / s : 0;
}

// Phase 1 (section 4.2, eqs. 13-15): coarse histogram of the view
// V = {i < L : i = a_r (mod s)} and the boundaries tau0 / tau1 with their
// inclusive cutoffs.  Entered with a cleared histogram; leaves it dirty.
template <int THREADS>
__device__ void sample_view(const Params& p, const float* row, int L, int a, RowState& st) {
  for (int t = threadIdx.x;; t += THREADS) {
    const int64_t i = (int64_t)a + (int64_t)t * p.s;
    if (i >= L) break;
    const uint32_t u = ld_stream1(row + i);
    atomicAdd(&st.hist[coarse_bin(u, desc_key(u))], 1u);
  }
  __syncthreads();
  find_boundaries<THREADS>(st, 2048, 2, (uint32_t)p.q0, (uint32_t)p.q1);
  const int tid = threadIdx.x;
  if (tid == 0) st.cut[0] = cutoff_for_bin(st.res_bin[0]);
  if (tid == 32 && p.dual) st.cut[1] = cutoff_for_bin(st.res_bin[1]);
  __syncthreads();
}

// Optional guess source (previous-step Top-K): the worst coarse bin of the K
// guessed scores, valid only when all K entries are positions of this row.
template <int THREADS>
__device__ bool guess_bin(const Params& p, const float* row, int L, int r, RowState& st) {
  if (threadIdx.x == 0) {
    st.gmax = -1;
    st.ginvalid = 0;
  }
  __syncthreads();
  const int32_t* g = p.prev + (int64_t)r * p.K;
  int worst = -1, invalid = 0;
  for (int t = threadIdx.x; t < p.K; t += THREADS) {
    const int32_t idx = g[t];
    if (idx < 0 || idx >= L) {
      invalid = 1;
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(row) + idx);
      worst = max(worst, coarse_bin(u, desc_key(u)));
    }
  }
  if (invalid) atomicOr(&st.ginvalid, 1);
  if (worst >= 0) atomicMax(&st.gmax, worst);
  __syncthreads();
  const bool ok = st.ginvalid == 0;
  if (ok && threadIdx.x == 0) st.cut[0] = cutoff_for_bin(st.gmax);
  __syncthreads();
  return ok;
}

// One row on the persistent sampled body: Phases 1-3 with band rescue and
// exact recovery, all under one CTA (section 5.5, "Persistent sampled").
template <int THREADS>
__device__ void sampled_row(const Params& p, int r, const Frontier& F, RowState& st) {
  const int K = p.K;
  const float* row = p.logits + (int64_t)r * p.pitch;
  int L = p.ke[r];
  L = L < 0 ? 0 : (L > p.N ? p.N : L);
  int32_t* out_row = p.out + (int64_t)r * K;
  if (L <= K) {
    write_pad_row<THREADS>(out_row, L, K);
    write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    return;
  }
  clear_hist<THREADS>(st, 2048);
  if (threadIdx.x == 0) {
    st.n_front = 0u;
    st.n_out = 0u;
  }
  __syncthreads();

  int route = -1, tau0 = -1, tau1 = -1, c0 = -1, c1 = -1;
  bool certified = false;
  if (p.prev != nullptr && guess_bin<THREADS>(p, row, L, r, st)) {
    tau0 = st.gmax;
    scan_admit<THREADS>(row, 0, L, 0u, st.cut[0], F, st);
    __syncthreads();
    c0 = (int)st.n_front;
    certified = c0 >= K;
    route = certified ? EXACT_TOPK_ROUTE_GUESS : EXACT_TOPK_ROUTE_GUESS_EXACT;
  } else {
    const int a = view_phase(r, p.s, p.s_bits);
    const int nv = view_size(L, a, p.s);
    const int qmax = p.dual ? p.q1 : p.q0;
    if (nv >= qmax) {
      sample_view<THREADS>(p, row, L, a, st);
      tau0 = st.res_bin[0];
      tau1 = p.dual ? st.res_bin[1] : -1;
      const uint32_t T0 = st.cut[0], T1 = st.cut[1];
      clear_hist<THREADS>(st, 2048);
      __syncthreads();
      scan_admit<THREADS>(row, 0, L, 0u, T0, F, st);  // Phase 2
      __syncthreads();
      c0 = (int)st.n_front;
      if (c0 >= K) {
        route = EXACT_TOPK_ROUTE_PRIMARY;
        certified = true;
      } else if (p.dual) {
        // Band rescue (eqs. 18-19): append only T0 < d <= T1.
        if (T1 > T0) scan_admit<THREADS>(row, 0, L, T0 + 1u, T1 - T0 - 1u, F, st);
        __syncthreads();
        c1 = (int)st.n_front;
        certified = c1 >= K;
        route = certified ? EXACT_TOPK_ROUTE_BAND : EXACT_TOPK_ROUTE_EXACT_AFTER_BAND;
      } else {
        route = EXACT_TOPK_ROUTE_EXACT_NO_BAND;
      }
    } else {
      route = EXACT_TOPK_ROUTE_DIRECT_EXACT;
    }
  }
  int tstar = -1, e0 = 0, q0n;
  if (certified) {
    q0n = (int)st.n_front;  // eq. 21: E0 = {}, Q0 = A(tau), k0 = K, h0 = h0^(tau)
    refine<THREADS>(F, st.n_front, (uint32_t)K, st, out_row, K);
  } else {
    exact_route<THREADS>(p, row, L, F, st, out_row, tstar, e0, q0n);
  }
  finish_row<THREADS>(p, st, out_row);
  write_trace(p, r, route, tau0, tau1, c0, c1, tstar, e0, q0n);
}

// Last CTA out resets the queue head and the exit counter (section 5.5:
// "persistent counters are restored on device").
__device__ void exit_protocol(int32_t* counters) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(counters + kCtrExit, 1);
    if (prev == (int)(gridDim.x * gridDim.y) - 1) {
      atomicExch(counters + kCtrQueue, 0);
      atomicExch(counters + kCtrExit, 0);
    }
  }
}

__device__ __forceinline__ int live_rows(const Params& p) {
  int m = p.num_valid_rows ? *p.num_valid_rows : p.M_cap;
  return m < 0 ? 0 : (m > p.M_cap ? p.M_cap : m);
}

template <int THREADS>
__device__ __forceinline__ RowState& row_state() {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  return *reinterpret_cast<RowState*>(smem_raw);
}

template <int THREADS>
__device__ __forceinline__ Frontier make_frontier(const Params& p, int64_t slice) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Frontier F;
  F.s_idx = reinterpret_cast<int32_t*>(smem_raw + sizeof(RowState));
  F.s_key = reinterpret_cast<uint32_t*>(smem_raw + sizeof(RowState) + sizeof(int32_t) * p.cap);
  F.cap = (uint32_t)p.cap;
  if (p.ws_idx != nullptr) {
    F.g_idx = p.ws_idx + slice * p.N;
    F.g_key = p.ws_key + slice * p.N;
    F.gcap = (uint32_t)p.N;
  } else {
    F.g_idx = nullptr;
    F.g_key = nullptr;
    F.gcap = 0u;
  }
  return F;
}

// ----------------------------------------------------------------------------
// Kernel 1: persistent sampled
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(kPersistentThreads, 3) persistent_sampled_kernel(Params p) {
  RowState& st = row_state<kPersistentThreads>();
  const Frontier F = make_frontier<kPersistentThreads>(p, blockIdx.x);
  const int M = live_rows(p);
  int r = blockIdx.x;
  while (r < M) {
    sampled_row<kPersistentThreads>(p, r, F, st);
    __syncthreads();
    if (threadIdx.x == 0) st.next_row = (int)gridDim.x + atomicAdd(p.counters + kCtrQueue, 1);
    __syncthreads();
    r = st.next_row;
  }
  exit_protocol(p.counters);
}

// ----------------------------------------------------------------------------
// Kernel 2: row-local exact
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(kRowLocalThreads, 1) row_local_exact_kernel(Params p) {
  RowState& st = row_state<kRowLocalThreads>();
  const Frontier F = make_frontier<kRowLocalThreads>(p, blockIdx.x);
  const int M = live_rows(p);
  int r = blockIdx.x;
  while (r < M) {
    const int K = p.K;
    const float* row = p.logits + (int64_t)r * p.pitch;
    int L = p.ke[r];
    L = L < 0 ? 0 : (L > p.N ? p.N : L);
    int32_t* out_row = p.out + (int64_t)r * K;
    if (L <= K) {
      write_pad_row<kRowLocalThreads>(out_row, L, K);
      write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    } else {
      int tstar, e0, q0n;
      if (L <= kRowLocalResident)
        exact_route_resident<kRowLocalThreads, kRowLocalResident / kRowLocalThreads>(
            p, row, L, F, st, out_row, tstar, e0, q0n);
      else
        exact_route<kRowLocalThreads>(p, row, L, F, st, out_row, tstar, e0, q0n);
      finish_row<kRowLocalThreads>(p, st, out_row);
      write_trace(p, r, EXACT_TOPK_ROUTE_DIRECT_EXACT, -1, -1, -1, -1, tstar, e0, q0n);
    }
    __syncthreads();
    if (threadIdx.x == 0) st.next_row = (int)gridDim.x + atomicAdd(p.counters + kCtrQueue, 1);
    __syncthreads();
    r = st.next_row;
  }
  exit_protocol(p.counters);
}

// ----------------------------------------------------------------------------
// Kernel 3: KV-split sampled (section 4.5 eqs. 26-27; section 5.5)
// ----------------------------------------------------------------------------

// Segment p of a row of length L: contiguous, 4-float aligned starts.
__device__ __forceinline__ void segment_bounds(int L, int P, int p, int& lo, int& hi) {
  int seg = (L + P - 1) / P;
  seg = (seg + 3) & ~3;
  const int64_t a = (int64_t)p * seg;
  lo = a > L ? L : (int)a;
  const int64_t b = a + seg;
  hi = b > L ? L : (int)b;
}

__global__ void __launch_bounds__(kKvSplitThreads, 3) kv_split_kernel(Params p) {
  RowState& st = row_state<kKvSplitThreads>();
  const int r = blockIdx.y;
  const int seg = blockIdx.x;
  const int P = p.P;
  const int K = p.K;
  const int tid = threadIdx.x;
  if (r >= live_rows(p)) return;
  const float* row = p.logits + (int64_t)r * p.pitch;
  int L = p.ke[r];
  L = L < 0 ? 0 : (L > p.N ? p.N : L);
  int32_t* out_row = p.out + (int64_t)r * K;
  // Row buffer: segment-owned candidate ranges, later the finisher's spill.
  int32_t* rb_idx = p.ws_idx + (int64_t)r * p.N;
  uint32_t* rb_key = p.ws_key + (int64_t)r * p.N;
  Frontier F = make_frontier<kKvSplitThreads>(p, r);

  if (L <= K) {
    if (seg == 0) {
      write_pad_row<kKvSplitThreads>(out_row, L, K);
      write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    }
    return;
  }
  clear_hist<kKvSplitThreads>(st, 2048);
  if (tid == 0) {
    st.seg_c0 = 0u;
    st.seg_cb = 0u;
    st.n_front = 0u;
    st.n_out = 0u;
  }
  __syncthreads();

  // Every segment reconstructs the same row-local proposal from r alone.
  bool guess = false;
  int tau0 = -1, tau1 = -1;
  uint32_t T0 = 0u, T1 = 0u;
  bool use_band = false;
  if (p.prev != nullptr && guess_bin<kKvSplitThreads>(p, row, L, r, st)) {
    guess = true;
    tau0 = st.gmax;
    T0 = st.cut[0];
  } else {
    const int a = view_phase(r, p.s, p.s_bits);
    const int nv = view_size(L, a, p.s);
    const int qmax = p.dual ? p.q1 : p.q0;
    if (nv < qmax) {
      // View unusable: the row takes the direct-exact route on one CTA.
      if (seg == 0) {
        int tstar, e0, q0n;
        exact_route<kKvSplitThreads>(p, row, L, F, st, out_row, tstar, e0, q0n);
        finish_row<kKvSplitThreads>(p, st, out_row);
        write_trace(p, r, EXACT_TOPK_ROUTE_DIRECT_EXACT, -1, -1, -1, -1, tstar, e0, q0n);
      }
      return;
    }
    sample_view<kKvSplitThreads>(p, row, L, a, st);
    tau0 = st.res_bin[0];
    tau1 = p.dual ? st.res_bin[1] : -1;
    T0 = st.cut[0];
    T1 = st.cut[1];
    use_band = p.dual && T1 > T0;
  }

  // Phase 2 over this segment: primary candidates fill the segment's range
  // from its start, band candidates (T0 < d <= T1) from its end, so the band
  // costs no second traversal.
  int lo, hi;
  segment_bounds(L, P, seg, lo, hi);
  for_each_in_range<kKvSplitThreads, 4>(row, lo, hi, [&](uint32_t u, int i) {
    const uint32_t d = desc_key(u);
    if (d <= T0) {
      const uint32_t q = atomicAdd(&st.seg_c0, 1u);
      rb_idx[lo + q] = i;
      rb_key[lo + q] = d;
    } else if (use_band && d <= T1) {
      const uint32_t q = atomicAdd(&st.seg_cb, 1u);
      rb_idx[hi - 1 - q] = i;
      rb_key[hi - 1 - q] = d;
    }
  });
  __threadfence();  // every writer publishes its candidates before the arrival
  __syncthreads();
  int32_t* counts = p.seg_counts + ((int64_t)r * P + seg) * 2;
  if (tid == 0) {
    counts[0] = (int32_t)st.seg_c0;
    counts[1] = (int32_t)st.seg_cb;
    __threadfence();
    const int prev = atomicAdd(p.counters + kCtrArriveBase + r, 1);
    st.is_last = prev == P - 1;
  }
  __syncthreads();
  if (!st.is_last) return;

  // ---- finisher: merge (eq. 27), certify, refine or recover ----
  __threadfence();
  if (tid == 0) atomicExch(p.counters + kCtrArriveBase + r, 0);
  uint32_t c0 = 0u, cb = 0u;
  for (int q = 0; q < P; ++q) {
    const int32_t* cq = p.seg_counts + ((int64_t)r * P + q) * 2;
    c0 += (uint32_t)__ldcg(cq);
    cb += (uint32_t)__ldcg(cq + 1);
  }
  int route;
  bool certified;
  bool with_band = false;
  if (guess) {
    certified = c0 >= (uint32_t)K;
    route = certified ? EXACT_TOPK_ROUTE_GUESS : EXACT_TOPK_ROUTE_GUESS_EXACT;
  } else if (c0 >= (uint32_t)K) {
    certified = true;
    route = EXACT_TOPK_ROUTE_PRIMARY;
  } else if (p.dual) {
    with_band = true;
    certified = c0 + cb >= (uint32_t)K;
    route = certified ? EXACT_TOPK_ROUTE_BAND : EXACT_TOPK_ROUTE_EXACT_AFTER_BAND;
  } else {
    certified = false;
    route = EXACT_TOPK_ROUTE_EXACT_NO_BAND;
  }
  const int c1 = with_band ? (int)(c0 + cb) : -1;
  int tstar = -1, e0 = 0, q0n;
  if (certified) {
    // Gather the runs (segment p's primary range, then its band range) into
    // the frontier, in order.  Logical position f maps to shared memory below
    // cap and to rb[f] above; every source position is >= the number of
    // entries gathered before it, so chunked in-place gathering never
    // overwrites an unread entry.
    const uint32_t total = with_band ? c0 + cb : c0;
    clear_hist<kKvSplitThreads>(st, 2048);
    __syncthreads();
    constexpr int R = 4;
    constexpr uint32_t CH = kKvSplitThreads * R;
    // run walk state per thread is recomputed per element: runs are few.
    for (uint32_t c = 0; c < total; c += CH) {
      int32_t idx[R];
      uint32_t key[R];
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const uint32_t g = c + k * kKvSplitThreads + tid;
        idx[k] = -2;
        if (g < total) {
          uint32_t base = 0;
          for (int q = 0; q < P; ++q) {
            const int32_t* cq = p.seg_counts + ((int64_t)r * P + q) * 2;
            const uint32_t n0 = (uint32_t)__ldcg(cq);
            const uint32_t nb = with_band ? (uint32_t)__ldcg(cq + 1) : 0u;
            if (g < base + n0 + nb) {
              int slo, shi;
              segment_bounds(L, P, q, slo, shi);
              const uint32_t off = g - base;
              // band entries occupy [shi - nb, shi); read them in ascending
              // order so that every source position is >= its logical index
              const int src = off < n0 ? slo + (int)off : shi - (int)nb + (int)(off - n0);
              idx[k] = __ldcg(rb_idx + src);
              key[k] = __ldcg(rb_key + src);
              break;
            }
            base += n0 + nb;
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < R; ++k) {
        if (idx[k] == -2) continue;
        F.put(c + k * kKvSplitThreads + tid, idx[k], key[k]);
        atomicAdd(&st.hist[key[k] >> 21], 1u);
      }
      __syncthreads();
    }
    q0n = (int)total;
    refine<kKvSplitThreads>(F, total, (uint32_t)K, st, out_row, K);
  } else {
    exact_route<kKvSplitThreads>(p, row, L, F, st, out_row, tstar, e0, q0n);
  }
  finish_row<kKvSplitThreads>(p, st, out_row);
  write_trace(p, r, route, tau0, guess ? -1 : tau1, (int)c0, c1, tstar, e0, q0n);
}

// Kernel attributes are set once per (device, kernel); later launches, which
// may be inside a stream capture, only launch.
constexpr int kMaxDevices = 64;
volatile int g_attr_smem[kMaxDevices][4];

template <class KernelT>
int set_attrs(KernelT kernel, int family, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && g_attr_smem[dev][family] >= (int)smem) return EXACT_TOPK_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  if (cached) g_attr_smem[dev][family] = (int)smem;
  return EXACT_TOPK_OK;
}

}  // namespace

size_t shared_bytes(int family, int cap) {
  (void)family;
  return sizeof(RowState) + (size_t)cap * (sizeof(int32_t) + sizeof(uint32_t));
}

int kernel_occupancy(int family, int device, int* ctas_per_sm) {
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  int rc = EXACT_TOPK_OK, n = 0;
  cudaError_t e = cudaSuccess;
  if (family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED) {
    const size_t smem = shared_bytes(family, kPersistentCap);
    rc = set_attrs(persistent_sampled_kernel, EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, smem);
    if (rc == EXACT_TOPK_OK)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, persistent_sampled_kernel,
                                                        kPersistentThreads, smem);
  } else if (family == EXACT_TOPK_FAMILY_KV_SPLIT) {
    const size_t smem = shared_bytes(family, kKvSplitCap);
    rc = set_attrs(kv_split_kernel, EXACT_TOPK_FAMILY_KV_SPLIT, smem);
    if (rc == EXACT_TOPK_OK)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kv_split_kernel, kKvSplitThreads, smem);
  } else {
    const size_t smem = shared_bytes(family, kRowLocalCap);
    rc = set_attrs(row_local_exact_kernel, EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT, smem);
    if (rc == EXACT_TOPK_OK)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, row_local_exact_kernel,
                                                        kRowLocalThreads, smem);
  }
  if (prev != device) cudaSetDevice(prev);
  if (rc != EXACT_TOPK_OK) return rc;
  if (e != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  *ctas_per_sm = n;
  return EXACT_TOPK_OK;
}

int launch(const exact_topk_plan& plan, const LaunchArgs& a, cudaStream_t stream) {
  const WorkspaceLayout lay = workspace_layout(plan);
  Params p;
  p.logits = a.logits;
  p.pitch = plan.row_pitch;
  p.N = (int32_t)plan.max_kv_len;
  p.M_cap = (int32_t)plan.num_rows;
  p.K = plan.top_k;
  p.s = plan.stride;
  int bits = 0;
  while ((1 << bits) < plan.stride) ++bits;
  p.s_bits = bits;
  p.dual = plan.dual;
  p.q0 = plan.q0;
  p.q1 = plan.q1;
  p.P = plan.splits;
  p.cap = plan.cand_capacity;
  p.ke = a.ke;
  p.out = a.out;
  p.num_valid_rows = a.num_valid_rows;
  p.counters = static_cast<int32_t*>(a.counters);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  if (lay.slices > 0 && ws != nullptr) {
    p.ws_idx = reinterpret_cast<int32_t*>(ws + lay.idx_offset);
    p.ws_key = reinterpret_cast<uint32_t*>(ws + lay.key_offset);
  } else {
    p.ws_idx = nullptr;
    p.ws_key = nullptr;
  }
  p.seg_counts = plan.family == EXACT_TOPK_FAMILY_KV_SPLIT
                     ? reinterpret_cast<int32_t*>(ws + lay.seg_offset)
                     : nullptr;
  p.prev = a.prev_topk;
  p.trace = a.trace;
  const size_t smem = shared_bytes(plan.family, plan.cand_capacity);
  int rc = EXACT_TOPK_OK;
  switch (plan.family) {
    case EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED:
      rc = set_attrs(persistent_sampled_kernel, EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, smem);
      if (rc != EXACT_TOPK_OK) return rc;
      persistent_sampled_kernel<<<plan.workers, kPersistentThreads, smem, stream>>>(p);
      break;
    case EXACT_TOPK_FAMILY_KV_SPLIT: {
      rc = set_attrs(kv_split_kernel, EXACT_TOPK_FAMILY_KV_SPLIT, smem);
      if (rc != EXACT_TOPK_OK) return rc;
      const dim3 grid((unsigned)plan.splits, (unsigned)plan.num_rows);
      kv_split_kernel<<<grid, kKvSplitThreads, smem, stream>>>(p);
      break;
    }
    case EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT:
      rc = set_attrs(row_local_exact_kernel, EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT, smem);
      if (rc != EXACT_TOPK_OK) return rc;
      row_local_exact_kernel<<<plan.workers, kRowLocalThreads, smem, stream>>>(p);
      break;
    default:
      return EXACT_TOPK_ERR_BAD_PLAN;
  }
  return cudaGetLastError() == cudaSuccess ? EXACT_TOPK_OK : EXACT_TOPK_ERR_CUDA;
}

}  // namespace etk

// ----------------------------------------------------------------------------
// Allocation-free entry point
// ----------------------------------------------------------------------------
//
// Some callers cannot allocate device memory at the point where they need a
// Top-K: code that runs while a stream capture is already open (a cudaMalloc
// there would invalidate the capture), plugins whose host framework owns every
// device allocation, and latency-critical loops where cudaMalloc's implicit
// device synchronization is unacceptable.  For them this entry point runs the
// KV-split kernel with its counters and workspace carved out of one file-scope
// device array instead of caller-provided buffers.

namespace etk {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // EXACT_TOPK_NOALLOC_SCRATCH_BYTES

// Loaded with the library's device code on every GPU that uses the library and
// kept until the process exits.  Shared by every call on that device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];
bool g_noalloc_have_info[kMaxDevices];
exact_topk_device_info g_noalloc_info[kMaxDevices];

// Once per device, with that device current: the device address of the
// scratch array (the host-side symbol is only a stand-in, never a device
// pointer) and the device facts the planner needs.
int noalloc_setup(int dev, void** ptr, exact_topk_device_info* info) {
  if (dev < 0 || dev >= kMaxDevices) return EXACT_TOPK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return EXACT_TOPK_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  if (!g_noalloc_have_info[dev]) {
    const int rc = exact_topk_query_device(dev, &g_noalloc_info[dev]);
    if (rc != EXACT_TOPK_OK) return rc;
    g_noalloc_have_info[dev] = true;
  }
  *ptr = g_noalloc_ptr[dev];
  *info = g_noalloc_info[dev];
  return EXACT_TOPK_OK;
}

}  // namespace
}  // namespace etk

extern "C" int exact_topk_kv_split_noalloc(const float* logits, int64_t num_rows,
                                           int64_t max_kv_len, const int32_t* ke, int32_t* out,
                                           const int32_t* num_valid_rows, int top_k,
                                           struct CUstream_st* stream) {
  using namespace etk;
  if (logits == nullptr || ke == nullptr || out == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  void* base = nullptr;
  exact_topk_device_info info;
  int rc = noalloc_setup(dev, &base, &info);
  if (rc != EXACT_TOPK_OK) return rc;
  exact_topk_plan_request req{};
  req.family = EXACT_TOPK_FAMILY_KV_SPLIT;
  req.dual = -1;
  exact_topk_plan plan;
  rc = exact_topk_make_plan(num_rows, max_kv_len, max_kv_len, top_k, &info, &req, &plan);
  if (rc != EXACT_TOPK_OK) return rc;
  const uint64_t ctr_bytes = (plan.counter_bytes + 255u) / 256u * 256u;
  if (ctr_bytes + plan.workspace_bytes > kNoAllocScratchBytes)
    return EXACT_TOPK_ERR_WORKSPACE_TOO_SMALL;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  // The array keeps whatever the previous call left; the counters must start
  // at zero, so clear them on the stream (a memset, not an allocation).
  if (cudaMemsetAsync(scratch, 0, (size_t)plan.counter_bytes,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  return exact_topk_run(&plan, logits, ke, out, num_valid_rows, scratch,
                        (size_t)plan.counter_bytes, scratch + ctr_bytes,
                        (size_t)plan.workspace_bytes, nullptr, nullptr, stream);
}
