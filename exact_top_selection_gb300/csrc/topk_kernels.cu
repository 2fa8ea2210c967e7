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
//
// Complete-row passes stream the row with 256-bit loads that carry an L2
// evict-first hint, so the lines the Phase-1 view touched (loaded with normal
// priority) tend to stay in L2 until the complete-row pass reaches them.  Each
// thread filters a tile of 16 scores with one max (or min) reduction; only
// tiles holding a candidate take the warp-aggregated append path.

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "etk_internal.h"

namespace etk {
namespace {

constexpr int kCoarseBins = 2048;
constexpr int kMaxSplits = 128;
// Resident CTAs per SM the sampled kernels are compiled for (register budget).
#ifndef ETK_SAMPLED_MIN_CTAS
#define ETK_SAMPLED_MIN_CTAS 2
#endif
// 256-bit loads per thread per tile of a complete-row pass.
#ifndef ETK_TILE_V8
#define ETK_TILE_V8 2
#endif
// L2 eviction hint of complete-row loads: 1 = evict first, 0 = none.
#ifndef ETK_L2_EVICT_FIRST
#define ETK_L2_EVICT_FIRST 1
#endif
constexpr int kTileV8 = ETK_TILE_V8;
constexpr int kTileScores = 8 * kTileV8;
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

__device__ __forceinline__ int coarse_bin(uint32_t u) { return coarse_bin(u, desc_key(u)); }

// Largest kappa_down32 key whose coarse bin is <= tau: the inclusive FP32
// endpoint of the admitted prefix (section 4.3; section 5.2 "converts the
// selected bins to their inclusive FP32 endpoints").  c is non-decreasing along
// the key space, so a search finds it; the 32 lanes of one warp test 32
// evenly spaced keys per step, shrinking the interval ~33-fold.  Must be
// called by all 32 lanes of a warp; every lane returns the result.
__device__ uint32_t cutoff_for_bin_warp(int tau) {
  const int lane = threadIdx.x & 31;
  uint32_t lo = 0u, hi = 0xFFFFFFFFu;  // c(lo) <= tau for tau >= 0; answer in [lo, hi]
  while (lo < hi) {
    const uint32_t n = hi - lo;
    // 32 test points lo + (l + 1) * step, clamped to hi: non-decreasing in l.
    const uint32_t step = n <= 32u ? 1u : (uint32_t)(((uint64_t)n + 31u) >> 5);
    const uint64_t pp = (uint64_t)lo + (uint64_t)(lane + 1) * step;
    const uint32_t p = pp > hi ? hi : (uint32_t)pp;
    const bool ok = coarse_bin(bits_from_desc(p), p) <= tau;
    const unsigned m = __ballot_sync(kFull, ok);
    const int k = __popc(m);  // passing lanes form a prefix
    if (k == 0) {
      hi = __shfl_sync(kFull, p, 0) - 1u;
    } else {
      const uint32_t pk = __shfl_sync(kFull, p, k & 31);
      lo = __shfl_sync(kFull, p, k - 1);
      if (k < 32) hi = pk - 1u;
    }
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

// 256-bit streaming load of 8 score bit patterns (32-byte aligned address),
// read once per complete-row pass: no L1 allocation, evict first from L2.
__device__ __forceinline__ void ld_stream8(const float* p, uint32_t* x) {
#if ETK_L2_EVICT_FIRST
  asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
        "=r"(x[7])
      : "l"(p));
#else
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
        "=r"(x[7])
      : "l"(p));
#endif
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
  uint32_t hist[kCoarseBins];   // h_{r,s} -> h0 (Fig. 5); refinement alternates with hist2
  uint32_t hist2[kCoarseBins];
  uint32_t warp_sums[32];
  uint32_t run_pre[kMaxSplits + 1];  // KV-split finisher: run prefix over segments
  uint32_t run_c0[kMaxSplits];       // KV-split finisher: primary count per segment
  uint32_t run_cb[kMaxSplits];       // KV-split finisher: band count per segment
  int32_t res_bin[2];
  uint32_t res_below[2];
  uint32_t res_cnt[2];
  uint32_t n_front;  // frontier entries
  uint32_t n_out;    // output slots used
  uint32_t n_keep;   // survivors during an in-place compaction
  uint32_t n_drop;   // sink for counts that are not kept
  uint32_t cut[2];   // kappa_down32 cutoffs
  int32_t gmax;      // guess source: worst coarse bin
  int32_t ginvalid;  // guess source: an entry outside [0, L)
  int32_t next_row;
  int32_t is_last;
  uint32_t seg_c0;   // KV-split: this segment's primary candidates
  uint32_t seg_cb;   // KV-split: this segment's band candidates
  uint32_t tot_c0;   // KV-split finisher: merged counts
  uint32_t tot_cb;
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
  uint2* ws;            // [slices][N] (index, key) pairs
  int32_t* seg_counts;  // [M_cap][P][2]
  const int32_t* prev;
  int32_t* trace;
};

// Candidate frontier: logical entries [0, cap) live in shared memory, entries
// at logical positions >= cap live at the same position of a global slice of
// capacity gcap (section 5.4: "Two global ping-pong slices extend the shared
// frontier"; here one slice suffices because compaction is done in place).
// Entries are (index, key) pairs stored together.
struct Frontier {
  uint2* s;
  uint32_t cap;
  uint2* g;
  uint32_t gcap;

  __device__ __forceinline__ void put(uint32_t p, int32_t i, uint32_t d) const {
    if (p < cap)
      s[p] = make_uint2((uint32_t)i, d);
    else if (p < gcap)
      g[p] = make_uint2((uint32_t)i, d);
  }
  __device__ __forceinline__ void get(uint32_t p, int32_t& i, uint32_t& d) const {
    uint2 e = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
    if (p < cap)
      e = s[p];
    else if (p < gcap)
      e = __ldcg(g + p);
    i = (int32_t)e.x;
    d = e.y;
  }
};

// Dynamic shared memory: RowState, then cap frontier pairs, then one
// candidate-vector stack per warp.
__device__ __forceinline__ uint32_t* queue_area(const Params& p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  return reinterpret_cast<uint32_t*>(smem_raw + sizeof(RowState) + sizeof(uint2) * (size_t)p.cap);
}

__device__ __forceinline__ void flag_status(int32_t* counters, int bit) {
  atomicOr(counters + kCtrStatus, bit);
}

template <int THREADS>
__device__ __forceinline__ void clear_hist(RowState& st, int nbins) {
  for (int b = threadIdx.x; b < nbins; b += THREADS) st.hist[b] = 0u;
}

// For each target t (ntargets <= 2): res_bin = min{b : H(b) >= t} over the
// inclusive prefix H of hist[0, nbins), res_below = H(b - 1) and res_cnt =
// hist[b]; res_bin = -1 (res_below = total) when the total is below t.  The
// histogram is only read.  Must be entered by the whole CTA after the
// histogram is complete, with a barrier between consecutive calls (results of
// a call are written exactly once, by the thread owning the boundary bin or
// by the last thread); results are visible to every thread on return.
template <int THREADS>
__device__ void find_boundaries_in(const uint32_t* hist, RowState& st, int nbins, int ntargets,
                                   uint32_t t0, uint32_t t1) {
  constexpr int kWarps = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins / THREADS;  // nbins is 1024 or 2048, THREADS 512 or 1024
  const int b0 = tid * per;
  uint32_t local = 0;
  for (int k = 0; k < per; ++k) local += hist[b0 + k];
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) st.warp_sums[warp] = incl;
  __syncthreads();
  // Every warp scans the warp totals itself (no second barrier).
  uint32_t w = lane < kWarps ? st.warp_sums[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(kFull, w, o);
    if (lane >= o) w += v;
  }
  const uint32_t before_warp = warp ? __shfl_sync(kFull, w, warp - 1) : 0u;
  const uint32_t grand = __shfl_sync(kFull, w, kWarps - 1);
  uint32_t run = before_warp + (incl - local);
  for (int k = 0; k < per; ++k) {
    const uint32_t h = hist[b0 + k];
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
  if (tid == THREADS - 1) {
    if (grand < t0) {
      st.res_bin[0] = -1;
      st.res_below[0] = grand;
      st.res_cnt[0] = 0u;
    }
    if (ntargets > 1 && grand < t1) {
      st.res_bin[1] = -1;
      st.res_below[1] = grand;
      st.res_cnt[1] = 0u;
    }
  }
  __syncthreads();
}

template <int THREADS>
__device__ __forceinline__ void find_boundaries(RowState& st, int nbins, int ntargets, uint32_t t0,
                                                uint32_t t1) {
  find_boundaries_in<THREADS>(st.hist, st, nbins, ntargets, t0, t1);
}

// ----------------------------------------------------------------------------
// Complete-row passes
// ----------------------------------------------------------------------------

// The 32-byte aligned body of row[lo, hi): [a0, a0 + 8 * nvec); the scalar
// head [lo, a0) and tail [a0 + 8 * nvec, hi) hold at most 7 scores each
// (section 5.3: wide loads on the aligned body, narrower paths for the rest).
struct Span {
  int a0;
  int nvec;
  int a_end;
};

__device__ __forceinline__ Span aligned_span(const float* row, int lo, int hi) {
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row + lo);
  int head = (int)(((32u - (uint32_t)(addr & 31u)) & 31u) >> 2);  // scores are 4-byte aligned
  if (head > hi - lo) head = hi - lo;
  Span s;
  s.a0 = lo + head;
  s.nvec = (hi - s.a0) >> 3;
  s.a_end = s.a0 + (s.nvec << 3);
  return s;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Per-warp stack of 8-score vectors that hold at least one admitted score:
// kQueueCap entries of 8 bit patterns plus the vector's index in the pass.
constexpr int kQueueCap = 32 + 32 * kTileV8;  // < 32 before a tile + one tile's pushes
constexpr int kQueueWords = kQueueCap * 9;

struct WarpQueue {
  uint32_t* vals;  // [kQueueCap][8]
  int32_t* vidx;   // [kQueueCap]
};

// One pass over row[lo, hi) that classifies every score by its key d into
//   class A: d <= TA            (only when A_ON)
//   class B: d <= TB otherwise  (TB >= TA)
// and hands each admitted (position, index, key) to sinkA / sinkB, where the
// position comes from the shared counter cntA / cntB.
//
// Streaming part, per thread: tiles of kTileV8 256-bit vectors, the next
// tile's loads issued before the current tile is filtered.  A vector is kept
// when its largest score passes (SIGNED_FAST: the cutoff TB is a non-negative
// score, so "d <= TB" is the signed compare (int)u >= (int)bits(TB) on the raw
// bits); one ballot per vector slot pushes the kept vectors onto the warp's
// stack.  Candidate part, per warp: whenever 32 vectors are stacked, each lane
// takes one, forms its admission mask, and the warp reserves positions with a
// scan and one shared atomic per class.  Candidate work therefore runs with
// full lanes instead of one lane per candidate.
template <int THREADS, bool SIGNED_FAST, bool A_ON, class SinkA, class SinkB>
__device__ __forceinline__ void drain_queue(const WarpQueue& q, int n, int a0, int CA, int CB,
                                            uint32_t TA, uint32_t TB, uint32_t* cntA,
                                            uint32_t* cntB, const SinkA& sinkA,
                                            const SinkB& sinkB) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = lanemask_lt();
  const int j = n - 32 + lane;  // n >= 32, or a final partial drain with n < 32
  const bool act = j >= 0;
  uint32_t u[8];
  int vi = 0;
  if (act) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(q.vals + 8 * j);
    const uint4 v1 = *reinterpret_cast<const uint4*>(q.vals + 8 * j + 4);
    u[0] = v0.x; u[1] = v0.y; u[2] = v0.z; u[3] = v0.w;
    u[4] = v1.x; u[5] = v1.y; u[6] = v1.z; u[7] = v1.w;
    vi = q.vidx[j];
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = SIGNED_FAST ? 0x80000000u : 0xFFFFFFFFu;
  }
  uint32_t m = 0u, mA = 0u;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const bool adm = SIGNED_FAST ? ((int)u[e] >= CB) : (act && desc_key(u[e]) <= TB);
    m |= adm ? (1u << e) : 0u;
    if (A_ON) {
      const bool a = SIGNED_FAST ? ((int)u[e] >= CA) : (desc_key(u[e]) <= TA);
      mA |= (adm && a) ? (1u << e) : 0u;
    }
  }
  const uint32_t mB = m & ~mA;
  const uint32_t packed = (uint32_t)__popc(mA) | ((uint32_t)__popc(mB) << 16);
  uint32_t incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t total = __shfl_sync(kFull, incl, 31);
  uint32_t bA = 0u, bB = 0u;
  if (lane == 0) {
    if (A_ON && (total & 0xFFFFu)) bA = atomicAdd(cntA, total & 0xFFFFu);
    if (total >> 16) bB = atomicAdd(cntB, total >> 16);
  }
  if (A_ON) bA = __shfl_sync(kFull, bA, 0);
  bB = __shfl_sync(kFull, bB, 0);
  const uint32_t excl = incl - packed;
  uint32_t pA = bA + (excl & 0xFFFFu), pB = bB + (excl >> 16);
  (void)lt;
  const int ibase = a0 + 8 * vi;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (m & (1u << e)) {
      const uint32_t d = desc_key(u[e]);
      if (A_ON && (mA & (1u << e)))
        sinkA(pA++, ibase + e, d);
      else
        sinkB(pB++, ibase + e, d);
    }
  }
}

template <int THREADS, bool SIGNED_FAST, bool A_ON, class SinkA, class SinkB>
__device__ __forceinline__ void scan_tiles(const float* row, int lo, int hi, uint32_t TA,
                                           uint32_t TB, uint32_t* cntA, uint32_t* cntB,
                                           uint32_t* queues, const SinkA& sinkA,
                                           const SinkB& sinkB) {
  if (lo >= hi) return;
  const int tid = threadIdx.x, lane = tid & 31;
  const Span sp = aligned_span(row, lo, hi);
  const int head = sp.a0 - lo, tail = hi - sp.a_end;
  if (tid < head + tail) {
    const int i = tid < head ? lo + tid : sp.a_end + (tid - head);
    const uint32_t d = desc_key(ld_stream1(row + i));
    if (d <= TB) {
      if (A_ON && d <= TA)
        sinkA(atomicAdd(cntA, 1u), i, d);
      else
        sinkB(atomicAdd(cntB, 1u), i, d);
    }
  }
  const int CB = (int)bits_from_desc(TB);
  const int CA = (int)bits_from_desc(TA);
  const uint32_t lt = lanemask_lt();
  WarpQueue q;
  q.vals = queues + (tid >> 5) * kQueueWords;
  q.vidx = reinterpret_cast<int32_t*>(q.vals + kQueueCap * 8);
  int qn = 0;  // warp-uniform stack depth
  const float* body = row + sp.a0;
  constexpr int kStep = kTileV8 * THREADS;
  constexpr uint32_t kSentinel = SIGNED_FAST ? 0x80000000u : 0xFFFFFFFFu;
  uint32_t x[kTileScores];
#pragma unroll
  for (int g = 0; g < kTileV8; ++g) {
    const int idx = g * THREADS + tid;
    if (idx < sp.nvec) {
      ld_stream8(body + 8 * idx, &x[8 * g]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) x[8 * g + k] = kSentinel;
    }
  }
  for (int t = 0; t < sp.nvec; t += kStep) {
    uint32_t y[kTileScores];
    const bool more = t + kStep < sp.nvec;
#pragma unroll
    for (int g = 0; g < kTileV8; ++g) {
      const int idx = t + kStep + g * THREADS + tid;
      if (more && idx < sp.nvec) {
        ld_stream8(body + 8 * idx, &y[8 * g]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) y[8 * g + k] = kSentinel;
      }
    }
#pragma unroll
    for (int g = 0; g < kTileV8; ++g) {
      const int vi = t + g * THREADS + tid;
      bool keep;
      if (SIGNED_FAST) {
        int mx = (int)x[8 * g];
#pragma unroll
        for (int k = 1; k < 8; ++k) mx = max(mx, (int)x[8 * g + k]);
        keep = mx >= CB;
      } else {
        uint32_t mn = desc_key(x[8 * g]);
#pragma unroll
        for (int k = 1; k < 8; ++k) mn = min(mn, desc_key(x[8 * g + k]));
        keep = vi < sp.nvec && mn <= TB;
      }
      const uint32_t bal = __ballot_sync(kFull, keep);
      if (bal != 0u) {
        if (keep) {
          const int pos = qn + __popc(bal & lt);
          uint4* dst = reinterpret_cast<uint4*>(q.vals + 8 * pos);
          dst[0] = make_uint4(x[8 * g], x[8 * g + 1], x[8 * g + 2], x[8 * g + 3]);
          dst[1] = make_uint4(x[8 * g + 4], x[8 * g + 5], x[8 * g + 6], x[8 * g + 7]);
          q.vidx[pos] = vi;
        }
        qn += __popc(bal);
      }
    }
    if (qn >= 32) {
      __syncwarp();
      do {
        drain_queue<THREADS, SIGNED_FAST, A_ON>(q, qn, sp.a0, CA, CB, TA, TB, cntA, cntB, sinkA,
                                                sinkB);
        qn -= 32;
      } while (qn >= 32);
      __syncwarp();
    }
#pragma unroll
    for (int k = 0; k < kTileScores; ++k) x[k] = y[k];
  }
  if (qn > 0) {
    __syncwarp();
    drain_queue<THREADS, SIGNED_FAST, A_ON>(q, qn, sp.a0, CA, CB, TA, TB, cntA, cntB, sinkA,
                                            sinkB);
    __syncwarp();
  }
}

// Dispatches on the cutoff's sign (signed-compare fast path) and on whether
// class A exists.
template <int THREADS, class SinkA, class SinkB>
__device__ __forceinline__ void scan_two_class(const float* row, int lo, int hi, uint32_t TA,
                                               uint32_t TB, bool a_on, uint32_t* cntA,
                                               uint32_t* cntB, uint32_t* queues,
                                               const SinkA& sinkA, const SinkB& sinkB) {
  const bool fast = (bits_from_desc(TB) & 0x80000000u) == 0u;
  if (fast) {
    if (a_on)
      scan_tiles<THREADS, true, true>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
    else
      scan_tiles<THREADS, true, false>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
  } else {
    if (a_on)
      scan_tiles<THREADS, false, true>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
    else
      scan_tiles<THREADS, false, false>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
  }
}

// Coarse histogram over row[lo, hi) (first pass of exact coarse recovery, eq. 20).
template <int THREADS>
__device__ void scan_coarse_hist(const float* row, int lo, int hi, RowState& st) {
  if (lo >= hi) return;
  const int tid = threadIdx.x;
  const Span sp = aligned_span(row, lo, hi);
  const int head = sp.a0 - lo, tail = hi - sp.a_end;
  if (tid < head + tail) {
    const int i = tid < head ? lo + tid : sp.a_end + (tid - head);
    atomicAdd(&st.hist[coarse_bin(ld_stream1(row + i))], 1u);
  }
  const float* body = row + sp.a0;
  for (int t = tid; t < sp.nvec; t += 2 * THREADS) {
    uint32_t x[16];
    const bool second = t + THREADS < sp.nvec;
    ld_stream8(body + 8 * t, x);
    if (second) ld_stream8(body + 8 * (t + THREADS), x + 8);
#pragma unroll
    for (int k = 0; k < 8; ++k) atomicAdd(&st.hist[coarse_bin(x[k])], 1u);
    if (second) {
#pragma unroll
      for (int k = 8; k < 16; ++k) atomicAdd(&st.hist[coarse_bin(x[k])], 1u);
    }
  }
}

// Sinks: where an admitted (position, index, key) goes.
struct FrontierSink {  // frontier entry + leading-digit histogram (eqs. 17, 20)
  Frontier F;
  uint32_t* hist;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    F.put(p, i, d);
    atomicAdd(&hist[d >> 21], 1u);
  }
};
struct CommitSink {  // committed straight to the output (E0 of eq. 20)
  int32_t* out_row;
  uint32_t K;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t) const {
    if (p < K) out_row[p] = i;
  }
};
struct DropSink {
  __device__ __forceinline__ void operator()(uint32_t, int32_t, uint32_t) const {}
};

// Output slot reservation for one committed index.
__device__ __forceinline__ void commit(RowState& st, int32_t* out_row, int K, int32_t i) {
  const uint32_t slot = atomicAdd(&st.n_out, 1u);
  if (slot < (uint32_t)K) out_row[slot] = i;
}

// ----------------------------------------------------------------------------
// Phase 3: prefix-commit-retain refinement (section 4.4, eqs. 22-25)
// ----------------------------------------------------------------------------

// General form for frontiers that spill to global memory: in-place chunked
// compaction of the frontier at every digit.
// Entry: frontier holds n entries (Q0), st.hist holds h0 (digit 0 over Q0),
// k = k0 indices remain to be selected, st.n_out = |E0|.  Exit: st.n_out == K.
template <int THREADS>
__device__ void refine_general(const Frontier& F, uint32_t n, uint32_t k, RowState& st,
                               int32_t* out_row, int K) {
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

// Warp-aggregated commit of idx for the lanes where `com` holds.
__device__ __forceinline__ void commit_warp(RowState& st, int32_t* out_row, int K, bool com,
                                            int32_t idx, uint32_t lt) {
  const uint32_t bal = __ballot_sync(kFull, com);
  if (bal == 0u) return;
  uint32_t base = 0u;
  if ((threadIdx.x & 31) == 0) base = atomicAdd(&st.n_out, (uint32_t)__popc(bal));
  base = __shfl_sync(kFull, base, 0);
  if (com) {
    const uint32_t slot = base + (uint32_t)__popc(bal & lt);
    if (slot < (uint32_t)K) out_row[slot] = idx;
  }
}

// Phase 3 (section 4.4, eqs. 22-25) with the frontier resident in registers:
// each thread holds up to 8 (index, key) entries, so no entry moves between
// digits; the histogram of the next digit is built in a second buffer while
// the current digit is classified.  Same entry and exit conditions as
// refine_general, to which frontiers beyond shared memory are handed.
template <int THREADS>
__device__ void refine(const Frontier& F, uint32_t n, uint32_t k, RowState& st, int32_t* out_row,
                       int K) {
  constexpr int EPT = 8;
  if (n > F.cap || F.cap > (uint32_t)(EPT * THREADS)) {
    refine_general<THREADS>(F, n, k, st, out_row, K);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  uint32_t key[EPT];
  int32_t idx[EPT];
  uint32_t alive = 0u;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const uint32_t p = (uint32_t)(e * THREADS + tid);
    if (p < n) {
      const uint2 v = F.s[p];
      idx[e] = (int32_t)v.x;
      key[e] = v.y;
      alive |= 1u << e;
    } else {
      idx[e] = -1;
      key[e] = 0xFFFFFFFFu;
    }
  }
  uint32_t* hc = st.hist;
  uint32_t* hn = st.hist2;
  for (int q = tid; q < 2048; q += THREADS) hn[q] = 0u;
  __syncthreads();
  for (int j = 0; j < 3 && k > 0; ++j) {
    find_boundaries_in<THREADS>(hc, st, j == 2 ? 1024 : 2048, 1, k, 0u);
    const int b = st.res_bin[0];
    const uint32_t below = st.res_below[0], cnt = st.res_cnt[0];
    if (b < 0) {  // inconsistent counts: cannot happen; finish_row flags it
      k = 0;
      break;
    }
    // b_j = min{b : H_j(b) >= k_j} (eq. 23); commit digit < b_j (eq. 24), keep
    // digit == b_j (eq. 25).  When H_j(b_j) == k_j the boundary group closes
    // the quota and is committed too.
    const bool last = below + cnt == k;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const bool al = (alive >> e) & 1u;
      const int dg = (int)digit(key[e], j);
      const bool com = al && (last ? dg <= b : dg < b);
      const bool keep = al && !last && dg == b;
      commit_warp(st, out_row, K, com, idx[e], lt);
      if (keep && j < 2) atomicAdd(&hn[digit(key[e], j + 1)], 1u);
      if (!keep) alive &= ~(1u << e);
    }
    if (last) {
      k = 0;
      break;
    }
    k -= below;
    __syncthreads();  // next histogram complete; the finder is done with hc
    uint32_t* t = hc;
    hc = hn;
    hn = t;
    if (j < 1)
      for (int q = tid; q < 2048; q += THREADS) hn[q] = 0u;  // ordered by the next finder's barrier
  }
  if (k > 0) {
    // After the last digit every alive key is identical: take the first k in
    // (thread, slot) order.
    const uint32_t c = (uint32_t)__popc(alive);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) st.warp_sums[warp] = incl;
    __syncthreads();
    uint32_t w = lane < THREADS / 32 ? st.warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += v;
    }
    uint32_t rank = (warp ? __shfl_sync(kFull, w, warp - 1) : 0u) + incl - c;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const bool al = (alive >> e) & 1u;
      commit_warp(st, out_row, K, al && rank < k, idx[e], lt);
      rank += al ? 1u : 0u;
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

// Cutoffs of the exact coarse boundary tau* (warps 0 and 1 in parallel):
// cut[1] admits c <= tau*, cut[0] admits c < tau* (none when tau* == 0).
template <int THREADS>
__device__ void exact_cutoffs(RowState& st, int tstar) {
  const int warp = threadIdx.x >> 5;
  if (warp == 0) {
    const uint32_t t = cutoff_for_bin_warp(tstar);
    if ((threadIdx.x & 31) == 0) st.cut[1] = t;
  } else if (warp == 1) {
    const uint32_t t = tstar > 0 ? cutoff_for_bin_warp(tstar - 1) : 0u;
    if ((threadIdx.x & 31) == 0) st.cut[0] = t;
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
  exact_cutoffs<THREADS>(st, tstar);
  const uint32_t tlo = st.cut[0], thi = st.cut[1];
  clear_hist<THREADS>(st, 2048);
  __syncthreads();
  CommitSink commit_sink{out_row, (uint32_t)K};
  FrontierSink front_sink{F, st.hist};
  scan_two_class<THREADS>(row, 0, L, tlo, thi, tstar > 0, &st.n_out, &st.n_front, queue_area(p), commit_sink,
                          front_sink);
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
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 31u) == 0u;
#pragma unroll
  for (int g = 0; g < VPT / 8; ++g) {
    const int i0 = (g * THREADS + tid) * 8;
    if (aligned && i0 + 7 < L) {
      ld_stream8(row + i0, v + 8 * g);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[g * 8 + e] = (i0 + e < L) ? ld_stream1(row + i0 + e) : 0u;
    }
  }
  clear_hist<THREADS>(st, 2048);
  if (tid == 0) {
    st.n_front = 0u;
    st.n_out = 0u;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < VPT / 8; ++g) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = (g * THREADS + tid) * 8 + e;
      if (i < L) atomicAdd(&st.hist[coarse_bin(v[g * 8 + e])], 1u);
    }
  }
  __syncthreads();
  find_boundaries<THREADS>(st, 2048, 1, (uint32_t)K, 0u);
  tstar = st.res_bin[0];
  e0 = (int)st.res_below[0];
  exact_cutoffs<THREADS>(st, tstar);
  clear_hist<THREADS>(st, 2048);
  __syncthreads();
  const uint32_t tlo = st.cut[0], thi = st.cut[1];
  const bool has_lo = tstar > 0;
#pragma unroll
  for (int g = 0; g < VPT / 8; ++g) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = (g * THREADS + tid) * 8 + e;
      if (i < L) {
        const uint32_t d = desc_key(v[g * 8 + e]);
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
// inclusive cutoffs.  Each thread issues up to 8 view loads before using any.
// Entered with a cleared histogram; leaves it dirty.
template <int THREADS>
__device__ void sample_view(const Params& p, const float* row, int L, int a, RowState& st) {
  const int nv = view_size(L, a, p.s);
  const int tid = threadIdx.x;
  for (int t0 = 0; t0 < nv; t0 += 8 * THREADS) {
    uint32_t u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = t0 + k * THREADS + tid;
      u[k] = t < nv ? __ldg(reinterpret_cast<const unsigned int*>(row) + a + (int64_t)t * p.s) : 0u;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t0 + k * THREADS + tid < nv) atomicAdd(&st.hist[coarse_bin(u[k])], 1u);
  }
  __syncthreads();
  find_boundaries<THREADS>(st, 2048, 2, (uint32_t)p.q0, (uint32_t)p.q1);
  const int warp = tid >> 5;
  if (warp == 0) {
    const uint32_t t = cutoff_for_bin_warp(st.res_bin[0]);
    if ((tid & 31) == 0) st.cut[0] = t;
  } else if (warp == 1 && p.dual) {
    const uint32_t t = cutoff_for_bin_warp(st.res_bin[1]);
    if ((tid & 31) == 0) st.cut[1] = t;
  }
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
      worst = max(worst, coarse_bin(u));
    }
  }
  if (invalid) atomicOr(&st.ginvalid, 1);
  if (worst >= 0) atomicMax(&st.gmax, worst);
  __syncthreads();
  const bool ok = st.ginvalid == 0;
  if (ok && threadIdx.x < 32) {
    const uint32_t t = cutoff_for_bin_warp(st.gmax);
    if (threadIdx.x == 0) st.cut[0] = t;
  }
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
    st.n_drop = 0u;
  }
  __syncthreads();

  FrontierSink front_sink{F, st.hist};
  DropSink drop;
  int route = -1, tau0 = -1, tau1 = -1, c0 = -1, c1 = -1;
  bool certified = false;
  if (p.prev != nullptr && guess_bin<THREADS>(p, row, L, r, st)) {
    tau0 = st.gmax;
    const uint32_t T = st.cut[0];
    scan_two_class<THREADS>(row, 0, L, T, T, false, &st.n_drop, &st.n_front, queue_area(p), drop,
                            front_sink);
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
      // Phase 2: admit d <= T0, persist candidates, build h0 (eqs. 16-17).
      scan_two_class<THREADS>(row, 0, L, T0, T0, false, &st.n_drop, &st.n_front, queue_area(p),
                              drop, front_sink);
      __syncthreads();
      c0 = (int)st.n_front;
      if (c0 >= K) {
        route = EXACT_TOPK_ROUTE_PRIMARY;
        certified = true;
      } else if (p.dual) {
        // Band rescue (eqs. 18-19): a second pass appends only T0 < d <= T1.
        if (T1 > T0)
          scan_two_class<THREADS>(row, 0, L, T0, T1, true, &st.n_drop, &st.n_front, queue_area(p), drop,
                                  front_sink);
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

__device__ __forceinline__ RowState& row_state() {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  return *reinterpret_cast<RowState*>(smem_raw);
}

__device__ __forceinline__ Frontier make_frontier(const Params& p, int64_t slice) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Frontier F;
  F.s = reinterpret_cast<uint2*>(smem_raw + sizeof(RowState));
  F.cap = (uint32_t)p.cap;
  if (p.ws != nullptr) {
    F.g = p.ws + slice * p.N;
    F.gcap = (uint32_t)p.N;
  } else {
    F.g = nullptr;
    F.gcap = 0u;
  }
  return F;
}

// ----------------------------------------------------------------------------
// Kernel 1: persistent sampled
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(kPersistentThreads, ETK_SAMPLED_MIN_CTAS) persistent_sampled_kernel(Params p) {
  RowState& st = row_state();
  const Frontier F = make_frontier(p, blockIdx.x);
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
  RowState& st = row_state();
  const Frontier F = make_frontier(p, blockIdx.x);
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

// Segment p of a row of length L: contiguous, starts 8-float (32-byte) aligned
// relative to the row start.
__device__ __forceinline__ void segment_bounds(int L, int P, int p, int& lo, int& hi) {
  int seg = (L + P - 1) / P;
  seg = (seg + 7) & ~7;
  const int64_t a = (int64_t)p * seg;
  lo = a > L ? L : (int)a;
  const int64_t b = a + seg;
  hi = b > L ? L : (int)b;
}

// Segment candidate sinks: primary entries fill the segment's range of the row
// buffer from its start, band entries from its end.
struct SegmentFrontSink {
  uint2* rb;
  int lo;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    rb[lo + (int)p] = make_uint2((uint32_t)i, d);
  }
};
struct SegmentBackSink {
  uint2* rb;
  int hi;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    rb[hi - 1 - (int)p] = make_uint2((uint32_t)i, d);
  }
};

__global__ void __launch_bounds__(kKvSplitThreads, ETK_SAMPLED_MIN_CTAS) kv_split_kernel(Params p) {
  RowState& st = row_state();
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
  uint2* rb = p.ws + (int64_t)r * p.N;
  const Frontier F = make_frontier(p, r);

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

  // Phase 2 over this segment, with the band (T0 < d <= T1) collected in the
  // same traversal: an underfilled primary needs no second pass.
  int lo, hi;
  segment_bounds(L, P, seg, lo, hi);
  {
    SegmentFrontSink primary{rb, lo};
    SegmentBackSink band{rb, hi};
    scan_two_class<kKvSplitThreads>(row, lo, hi, T0, use_band ? T1 : T0, true, &st.seg_c0,
                                    &st.seg_cb, queue_area(p), primary, band);
  }
  __threadfence();  // every writer publishes its candidates before the arrival
  __syncthreads();
  if (tid == 0) {
    int32_t* counts = p.seg_counts + ((int64_t)r * P + seg) * 2;
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
  for (int q = tid; q < P; q += kKvSplitThreads) {
    const int32_t* cq = p.seg_counts + ((int64_t)r * P + q) * 2;
    st.run_c0[q] = (uint32_t)__ldcg(cq);
    st.run_cb[q] = (uint32_t)__ldcg(cq + 1);
  }
  __syncthreads();
  if (tid < 32) {
    // Totals of both counts, each lane summing up to 4 consecutive segments.
    uint32_t s0 = 0u, sb = 0u;
    for (int q = tid * 4; q < tid * 4 + 4 && q < P; ++q) {
      s0 += st.run_c0[q];
      sb += st.run_cb[q];
    }
    s0 = __reduce_add_sync(kFull, s0);
    sb = __reduce_add_sync(kFull, sb);
    if (tid == 0) {
      st.tot_c0 = s0;
      st.tot_cb = sb;
    }
  }
  __syncthreads();
  const uint32_t c0 = st.tot_c0, cb = st.tot_cb;
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
    // Run table: segment q contributes its primary range then (band route)
    // its band range, in segment order.
    if (tid == 0) {
      uint32_t acc = 0u;
      for (int q = 0; q < P; ++q) {
        st.run_pre[q] = acc;
        acc += st.run_c0[q] + (with_band ? st.run_cb[q] : 0u);
      }
      st.run_pre[P] = acc;
    }
    clear_hist<kKvSplitThreads>(st, 2048);
    __syncthreads();
    // Gather the runs into the frontier in order.  Logical position f maps to
    // shared memory below cap and to rb[f] above; every source position is >=
    // its logical position, so gathering in chunks (read all, then write)
    // never overwrites an unread entry.
    const uint32_t total = st.run_pre[P];
    constexpr int R = 4;
    constexpr uint32_t CH = kKvSplitThreads * R;
    for (uint32_t c = 0; c < total; c += CH) {
      int32_t idx[R];
      uint32_t key[R];
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const uint32_t g = c + k * kKvSplitThreads + tid;
        idx[k] = -2;
        if (g < total) {
          int lo_q = 0, hi_q = P - 1;  // last q with run_pre[q] <= g
          while (lo_q < hi_q) {
            const int mid = (lo_q + hi_q + 1) >> 1;
            if (st.run_pre[mid] <= g)
              lo_q = mid;
            else
              hi_q = mid - 1;
          }
          const int q = lo_q;
          int slo, shi;
          segment_bounds(L, P, q, slo, shi);
          const uint32_t off = g - st.run_pre[q];
          const uint32_t n0 = st.run_c0[q];
          // band entries occupy [shi - nb, shi); read them in ascending order
          // so that every source position is >= its logical position
          const int src = off < n0 ? slo + (int)off
                                   : shi - (int)st.run_cb[q] + (int)(off - n0);
          const uint2 e = __ldcg(rb + src);
          idx[k] = (int32_t)e.x;
          key[k] = e.y;
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
  const int threads =
      family == EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT ? kRowLocalThreads : kPersistentThreads;
  return sizeof(RowState) + (size_t)cap * sizeof(uint2) +
         (size_t)(threads / 32) * kQueueWords * sizeof(uint32_t);
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
  p.ws = (lay.slices > 0 && ws != nullptr) ? reinterpret_cast<uint2*>(ws + lay.pair_offset)
                                            : nullptr;
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
      if (plan.splits > kMaxSplits) return EXACT_TOPK_ERR_BAD_PLAN;
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
