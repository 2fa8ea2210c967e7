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
//   cluster_split_kernel       the P CTAs of one thread-block cluster hold one
//                              row in shared memory (TMA bulk copies) and merge
//                              through distributed shared memory.
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
// priority) tend to stay in L2 until the complete-row pass reaches them.

#include <cuda.h>  // CUtensorMap and its encoder's types (the encoder is reached at run time)
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "etk_internal.h"

namespace etk {
namespace {

constexpr int kCoarseBins = 2048;
constexpr int kMaxSplits = 128;
// Depth of each thread's ring of 256-bit loads in a complete-row pass.  Two
// (one vector in flight while one is filtered) is the fastest on GB300: the
// persistent kernel runs at 64 registers a thread, every deeper slot holds
// eight more of them live across the filter (the causal prefill batch,
// 4096 rows of up to 131072 scores, takes 418 us at depth two, 434 us at
// three), and the TMA L2 prefetch ahead of the pass already keeps bytes in
// flight that hold no registers.
#ifndef ETK_RING
#define ETK_RING 2
#endif
constexpr int kRing = ETK_RING;
constexpr uint32_t kDescPosInf = 0x007FFFFFu;  // kappa_down32(+inf)
constexpr uint32_t kDescNegInf = 0xFF800000u;  // kappa_down32(-inf)
constexpr unsigned kFull = 0xFFFFFFFFu;

// ----------------------------------------------------------------------------
// Thread groups
// ----------------------------------------------------------------------------

// The whole CTA.
template <int THREADS>
struct CtaGroup {
  static constexpr int kThreads = THREADS;
  static constexpr int kWarps = THREADS / 32;
  static_assert(THREADS % 32 == 0 && kWarps <= 32, "whole warps, at most 32");
  __device__ __forceinline__ static int rank() { return (int)threadIdx.x; }
  __device__ __forceinline__ static void sync() { __syncthreads(); }
};

// Warps FIRST_WARP .. FIRST_WARP + THREADS/32 - 1 of the CTA, synchronised by
// the named barrier BAR (never 0, which __syncthreads uses).  Two such groups
// with different barriers run different phases at the same time; every
// function they call synchronises through G::sync() only.
template <int THREADS, int FIRST_WARP, int BAR>
struct SubGroup {
  static constexpr int kThreads = THREADS;
  static constexpr int kWarps = THREADS / 32;
  static_assert(THREADS % 32 == 0 && kWarps <= 32, "whole warps, at most 32");
  static_assert(BAR > 0 && BAR < 16, "a named barrier other than 0");
  __device__ __forceinline__ static int rank() { return (int)threadIdx.x - FIRST_WARP * 32; }
  __device__ __forceinline__ static void sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(THREADS) : "memory");
  }
};

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
// evenly spaced keys per step.  Must be called by all 32 lanes of a warp;
// every lane returns the result.
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

// Closed-form candidate for cutoff_for_bin: bin tau's smallest admitted half
// is the one with kappa_down16 = 32 tau + 31; an FP32 score rounds (to nearest,
// ties to even) to that half or above iff it is >= the midpoint between the
// half and its lower neighbour (the midpoint itself when the half's mantissa
// is even, the next FP32 value above it otherwise).  Returns the key of that
// smallest admitted score; callers verify it.
__device__ __forceinline__ uint32_t cutoff_candidate(int tau) {
  if (tau >= kCoarseBins - 1) return 0xFFFFFFFFu;
  if (tau >= (int)(0xFC00u >> 5)) return kDescNegInf;  // c(-inf): every number admitted
  const uint32_t D = 32u * (uint32_t)tau + 31u;
  const uint32_t h = (D & 0x8000u) ? D : (D ^ 0x7FFFu);
  if (h == 0x0000u) return desc_key(0u);  // +0: every non-negative score
  float mid;
  if (h == 0x7C00u) {
    mid = 65520.0f;  // between 65504 and +inf
  } else if (h == 0xFBFFu) {
    mid = -65520.0f;  // between -65504 and -inf
  } else {
    const uint32_t hlo = (h & 0x8000u) ? h + 1u : h - 1u;  // next smaller half
    const float v = __half2float(__ushort_as_half((unsigned short)h));
    const float vlo = __half2float(__ushort_as_half((unsigned short)hlo));
    mid = (v + vlo) * 0.5f;  // exact: both are halves
  }
  uint32_t m = __float_as_uint(mid);
  if (h & 1u) m = (m & 0x80000000u) ? m - 1u : m + 1u;  // odd half: ties go below
  return desc_key(m);
}

// Cutoff of bin tau for one thread: the closed-form candidate when it
// verifies as the largest key with c <= tau, else the warp search's answer
// (the warp-wide form is used by callers that hold a whole warp).
__device__ __forceinline__ bool cutoff_verified(int tau, uint32_t T) {
  if (coarse_bin(bits_from_desc(T), T) > tau) return false;
  if (T == 0xFFFFFFFFu) return true;
  return coarse_bin(bits_from_desc(T + 1u), T + 1u) > tau;
}

// Warp-wide cutoff: candidate first, search only if it does not verify.
__device__ __forceinline__ uint32_t cutoff_fast_warp(int tau) {
  const uint32_t T = cutoff_candidate(tau);
  const bool ok = tau >= 0 && cutoff_verified(tau, T);
  if (__all_sync(kFull, ok)) return T;
  return cutoff_for_bin_warp(tau);
}

// Digit j of the 11+11+10 split, most significant first (section 4.3).
__device__ __forceinline__ uint32_t digit(uint32_t d, int j) {
  return j == 0 ? (d >> 21) : (j == 1 ? ((d >> 10) & 0x7FFu) : (d & 0x3FFu));
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Per-thread run-length merging of histogram increments: consecutive adds to
// the same bin become one shared atomic.  Rows of few distinct values
// (constant rows, tie bands, signed zeros) would otherwise put every lane of a
// warp on one shared address.
// Shared-memory reduction add on a histogram that lives in this CTA's shared
// memory, issued in the shared state space (the pointer may reach a function
// as a generic address).
__device__ __forceinline__ void smem_add(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v)
               : "memory");
}

struct RunHist {
  uint32_t bin = 0u, cnt = 0u;
  __device__ __forceinline__ void add(uint32_t* hist, uint32_t b) {
    if (cnt != 0u && b != bin) {
      smem_add(&hist[bin], cnt);
      cnt = 0u;
    }
    bin = b;
    ++cnt;
  }
  __device__ __forceinline__ void flush(uint32_t* hist) {
    if (cnt != 0u) smem_add(&hist[bin], cnt);
    cnt = 0u;
  }
};

// ----------------------------------------------------------------------------
// Loads
// ----------------------------------------------------------------------------

// 256-bit streaming load of 8 score bit patterns (32-byte aligned address),
// read once per complete-row pass: no L1 allocation, evict first from L2.
__device__ __forceinline__ void ld_stream8(const float* p, uint32_t* x) {
  asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),
        "=r"(x[7])
      : "l"(p));
}

// 128-bit read-once load of 4 score bit patterns (16-byte aligned address).
__device__ __forceinline__ uint4 ldg_v4(const float* p) {
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

// L2 prefetch of [p, p + bytes) by the TMA engine: a hint with no completion
// to wait for.  p 16-byte aligned, bytes a positive multiple of 16, the range
// inside one allocation.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// Bytes of a row kept requested ahead of a complete-row pass, and of the next
// row's head requested during a row's refinement.  On the causal prefill
// batch (304 CTAs streaming at once) 64-96 KB ahead and 32-64 KB of the next
// row measured 389-390 us against 396 us for 128 KB and 128 KB: requests that
// run further ahead only queue behind the other CTAs' and take L2 space.
#ifndef ETK_L2_AHEAD_KB
#define ETK_L2_AHEAD_KB 80
#endif
#ifndef ETK_L2_NEXT_KB
#define ETK_L2_NEXT_KB 64
#endif
constexpr uint32_t kL2Ahead = ETK_L2_AHEAD_KB * 1024u;
constexpr uint32_t kL2Next = ETK_L2_NEXT_KB * 1024u;

// Requests row[0, L) into L2 ahead of a pass over a row that one CTA reads
// several times (one thread; 64 KB per request, 16-byte aligned range).
__device__ __forceinline__ void prefetch_row_l2(const float* row, int L) {
  const uintptr_t b = (reinterpret_cast<uintptr_t>(row) + 15u) & ~(uintptr_t)15u;
  const uintptr_t e = (reinterpret_cast<uintptr_t>(row) + (uintptr_t)L * 4u) & ~(uintptr_t)15u;
  for (uintptr_t a = b; a < e; a += 65536u) {
    const uintptr_t len = e - a < 65536u ? e - a : 65536u;
    prefetch_l2(reinterpret_cast<const void*>(a), (uint32_t)len);
  }
}

// ----------------------------------------------------------------------------
// Shared state
// ----------------------------------------------------------------------------

// Scratch of one thread group for block-wide scans and boundary search.
struct GroupScratch {
  uint32_t warp_sums[32];
  int32_t res_bin[2];
  uint32_t res_below[2];
  uint32_t res_cnt[2];
  int32_t gmax;      // guess source: worst coarse bin
  int32_t ginvalid;  // guess source: an entry outside [0, L)
  int32_t bcast;     // broadcast word
  int32_t bcast2;    // second broadcast word
};

// One row in flight: its proposal, counters and route record.
struct Slot {
  int32_t row;  // -1: no more rows
  int32_t L;
  int32_t route;
  uint32_t T0, T1;  // kappa_down32 cutoffs
  int32_t tau0, tau1;
  uint32_t n_front;  // frontier entries
  uint32_t n_out;    // output slots used
  uint32_t n_keep;   // survivors during an in-place compaction
  uint32_t n_drop;   // sink for counts that are not kept
  int32_t c0, c1, tstar, e0, q0n;
  uint32_t seg_c0, seg_cb;  // KV-split: this segment's counts
  int32_t is_last;
  uint32_t vcnt0;  // Phase 1: view entries in bins <= tau0
  uint32_t vcnt1;  // ... and in bins <= tau1
  int32_t pad_;
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
  int32_t* defer;       // persistent family: [M_cap][8] deferred-row records
  const int32_t* prev;
  int32_t* trace;
  // Persistent kernel: tiled tensor map over the scores seen as
  // [M_cap][N / s][s] (lines of s scores), whose column `a` of a row is that
  // row's view; a box of {4, view_box, 1} carries view_box consecutive view
  // entries (with the three scores that share their 16 bytes).  view_tma = 0:
  // the view is gathered with plain loads.
  int32_t view_tma;
  int32_t view_box;
  CUtensorMap view_map;
};

// Candidate frontier: logical entries [0, cap) live in shared memory, entries
// at logical positions >= cap live at the same position of a global slice of
// capacity gcap (section 5.4: "Two global ping-pong slices extend the shared
// frontier"; here one slice per row slot suffices because compaction is done
// in place).  Entries are (index, key) pairs stored together.
constexpr int kRefineBatch = 8;  // frontier entries per thread in flight in Phase 3 histograms
constexpr int kCommitBatch = 4;  // ... and in its final commit pass

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

// Per-warp stack of 8-score vectors that hold at least one admitted score:
// kQueueCap entries of 8 bit patterns plus the vector's index in the pass.
constexpr int kQueueCap = 64;  // < 32 before a vector slot + at most 32 pushed by it
constexpr int kQueueWords = kQueueCap * 9;
// Persistent kernel: warps [0, kRefineWarps) refine the row just classified
// while the remaining warps claim the next row and run its Phase 1.
// TMA view boxes of up to 256 view entries (4 KB each) per persistent CTA.
constexpr uint32_t kViewBoxes = 4;
// Six of sixteen warps: with the range-relative refinement (refine_fast) the
// next row's Phase 1 is the longer half of the tail; measured on the causal
// prefill batch, 2, 4, 6 and 8 warps gave 470, 435, 429 and 433 us.
#ifndef ETK_PREPARE_WARPS
#define ETK_PREPARE_WARPS (3 * kPersistentThreads / 256)
#endif
constexpr int kRefineWarps = kPersistentThreads / 32 - ETK_PREPARE_WARPS;
static_assert(kRefineWarps > 0 && kRefineWarps < kPersistentThreads / 32,
              "both groups need at least one warp");

// Rows one persistent CTA may hand to its own epilogue (heavy rows beyond
// these take the frontier route).
constexpr uint32_t kMaxOwnDeferred = 63;

// Dynamic shared memory layouts (byte offsets), one per kernel family.
struct SmemLayout {
  uint32_t slots;     // Slot[nslots]
  uint32_t scratch;   // GroupScratch[2]
  uint32_t hist;      // uint32[nslots][2048]
  uint32_t frontier;  // uint2[cap]
  uint32_t runs;      // KV-split run table, or 0
  uint32_t vbuf;      // persistent: TMA view boxes, kViewBoxes x 4 KB (128-byte aligned), or 0
  uint32_t vbar;      // persistent: the view copies' mbarrier, and its phase word, or 0
  uint32_t own;       // persistent: count and indices of the rows this CTA deferred, or 0
  uint32_t queues;    // uint32[warps][kQueueWords]
  uint32_t total;
};

__host__ __device__ constexpr uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

// constexpr: each kernel passes its family's fixed candidate capacity, so the
// offsets are compile-time constants.
__host__ __device__ constexpr SmemLayout smem_layout(int family, int cap) {
  SmemLayout l{};
  const bool pers = family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED;
  // persistent: a second slot and histogram hold the next row's Phase 1
  const int nslots = pers ? 2 : 1;
  const int qwarps = pers ? kPersistentThreads / 32
                          : (family == EXACT_TOPK_FAMILY_KV_SPLIT ? kKvSplitThreads / 32
                                                                  : kRowLocalThreads / 32);
  uint32_t o = 0;
  l.slots = o;
  o = align16(o + nslots * (uint32_t)sizeof(Slot));
  l.scratch = o;
  o = align16(o + 2 * (uint32_t)sizeof(GroupScratch));
  l.hist = o;
  o = align16(o + nslots * kCoarseBins * 4u);
  l.frontier = o;
  o = align16(o + (uint32_t)cap * 8u);
  l.runs = family == EXACT_TOPK_FAMILY_KV_SPLIT ? o : 0u;
  if (family == EXACT_TOPK_FAMILY_KV_SPLIT) o = align16(o + (3 * kMaxSplits + 1) * 4u);
  l.vbuf = 0u;
  l.vbar = 0u;
  if (pers) {
    o = (o + 127u) & ~127u;
    l.vbuf = o;
    o += kViewBoxes * 4096u;
    l.vbar = o;
    o = align16(o + 16u);
    l.own = o;
    o = align16(o + (1u + kMaxOwnDeferred) * 4u);
  }
  l.queues = o;
  o = align16(o + qwarps * kQueueWords * 4u);
  l.total = o;
  return l;
}

__device__ __forceinline__ unsigned char* smem_base() {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  return smem_raw;
}

__device__ __forceinline__ void flag_status(int32_t* counters, int bit) {
  atomicOr(counters + kCtrStatus, bit);
}

template <class G>
__device__ __forceinline__ void clear_hist(uint32_t* hist, int nbins) {
  for (int b = G::rank(); b < nbins; b += G::kThreads) hist[b] = 0u;
}

// For each target t (ntargets <= 2): res_bin = min{b : H(b) >= t} over the
// inclusive prefix H of hist[0, nbins), res_below = H(b - 1) and res_cnt =
// hist[b]; res_bin = -1 (res_below = total) when the total is below t.  The
// histogram is only read.  Entered by the whole group after the histogram is
// complete, with a group barrier between consecutive calls; results are
// visible to every thread of the group on return.
//
// nbins is a multiple of 128 (at most 2048): warp w sums 128-bin chunks w,
// w + warps, ... (lane l holds bins 4l .. 4l+3 of a chunk), and after one
// barrier every warp scans the chunk totals, so that the warp whose chunk
// holds a target resolves it from the registers it already has.
template <class G>
__device__ void find_boundaries(const uint32_t* hist, GroupScratch& sc, int nbins, int ntargets,
                                uint32_t t0, uint32_t t1) {
  constexpr int kCpw = (16 + G::kWarps - 1) / G::kWarps;  // chunks per warp (nbins <= 2048)
  const int tid = G::rank(), lane = tid & 31, warp = tid >> 5;
  const int nch = nbins >> 7;
  uint4 v[kCpw];
  uint32_t s4[kCpw];
#pragma unroll
  for (int c = 0; c < kCpw; ++c) {
    const int ch = warp + c * G::kWarps;
    v[c] = make_uint4(0u, 0u, 0u, 0u);
    s4[c] = 0u;
    if (ch < nch) {
      v[c] = reinterpret_cast<const uint4*>(hist)[ch * 32 + lane];
      s4[c] = v[c].x + v[c].y + v[c].z + v[c].w;
      const uint32_t tot = __reduce_add_sync(kFull, s4[c]);
      if (lane == 0) sc.warp_sums[ch] = tot;
    }
  }
  G::sync();
  if (warp < nch) {
    const uint32_t ct = lane < nch ? sc.warp_sums[lane] : 0u;
    uint32_t cincl = ct;  // inclusive prefix over chunks
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, cincl, o);
      if (lane >= o) cincl += y;
    }
    const uint32_t grand = __shfl_sync(kFull, cincl, 31);
#pragma unroll
    for (int c = 0; c < kCpw; ++c) {
      const int ch = warp + c * G::kWarps;
      if (ch >= nch) break;  // warp-uniform
      const uint32_t before = __shfl_sync(kFull, cincl - ct, ch);  // before chunk ch
      uint32_t incl = s4[c];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = before + incl - s4[c];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (x >= ntargets) break;
        const uint32_t t = x == 0 ? t0 : t1;
        if (grand < t) {
          if (warp == 0 && c == 0 && lane == 0) {
            sc.res_bin[x] = -1;
            sc.res_below[x] = grand;
            sc.res_cnt[x] = 0u;
          }
          continue;
        }
        if (t == 0u) {  // H(0) >= 0
          if (warp == 0 && c == 0 && lane == 0) {
            sc.res_bin[x] = 0;
            sc.res_below[x] = 0u;
            sc.res_cnt[x] = hist[0];
          }
          continue;
        }
        // the lane (of the chunk's warp) whose four bins cross t
        if (excl < t && t <= excl + s4[c]) {
          const uint32_t h[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
          uint32_t r0 = excl;
          int b = -1;
          uint32_t bl = 0u, bc = 0u;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (b < 0 && r0 + h[i] >= t) {
              b = i;
              bl = r0;
              bc = h[i];
            }
            r0 += h[i];
          }
          sc.res_bin[x] = ch * 128 + lane * 4 + b;
          sc.res_below[x] = bl;
          sc.res_cnt[x] = bc;
        }
      }
    }
  }
  G::sync();
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

struct WarpQueue {
  uint32_t* vals;  // [kQueueCap][8]
  int32_t* vidx;   // [kQueueCap]
};

// Processes the top min(n, 32) stacked vectors: each lane takes one, forms
// its admission masks, and the warp reserves positions with a scan and one
// shared atomic per class.
template <bool SIGNED_FAST, bool A_ON, class SinkA, class SinkB>
__device__ __forceinline__ void drain_queue(const WarpQueue& q, int n, int a0, int CA, int CB,
                                            uint32_t TA, uint32_t TB, uint32_t* cntA,
                                            uint32_t* cntB, const SinkA& sinkA,
                                            const SinkB& sinkB) {
  const int lane = threadIdx.x & 31;
  const int j = n - 32 + lane;  // n >= 32, or a final partial drain with n < 32
  const bool act = j >= 0;
  uint32_t u[8];
  int vi = 0;
  if (act) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(q.vals + 8 * j);
    const uint4 v1 = *reinterpret_cast<const uint4*>(q.vals + 8 * j + 4);
    u[0] = v0.x;
    u[1] = v0.y;
    u[2] = v0.z;
    u[3] = v0.w;
    u[4] = v1.x;
    u[5] = v1.y;
    u[6] = v1.z;
    u[7] = v1.w;
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
  sinkA.count8(mA, u);
  sinkB.count8(mB, u);
}

// One pass of group G over row[lo, hi) that classifies every score by its
// key d into
//   class A: d <= TA            (only when A_ON)
//   class B: d <= TB otherwise  (TB >= TA)
// and hands each admitted (position, index, key) to sinkA / sinkB, where the
// position comes from the shared counter cntA / cntB.  No group barrier.
//
// Streaming part, per thread: a ring of kRing 256-bit vectors, kRing - 1 of
// them in flight while one is filtered.  A vector is kept
// when its largest score passes (SIGNED_FAST: the cutoff TB is a non-negative
// score, so "d <= TB" is the signed compare (int)u >= (int)bits(TB) on the raw
// bits); one ballot per vector slot pushes the kept vectors onto the warp's
// stack.  Candidate part, per warp: whenever 32 vectors are stacked, each
// lane takes one, so candidate work runs with full lanes instead of one lane
// per candidate.
template <class G, bool SIGNED_FAST, bool A_ON, class SinkA, class SinkB>
__device__ __forceinline__ void scan_tiles(const float* row, int lo, int hi, uint32_t TA,
                                           uint32_t TB, uint32_t* cntA, uint32_t* cntB,
                                           uint32_t* queues, const SinkA& sinkA,
                                           const SinkB& sinkB) {
  if (lo >= hi) return;
  const int tid = G::rank();
  const Span sp = aligned_span(row, lo, hi);
  const int head = sp.a0 - lo, tail = hi - sp.a_end;
  if (tid < head + tail) {
    const int i = tid < head ? lo + tid : sp.a_end + (tid - head);
    const uint32_t d = desc_key(ld_stream1(row + i));
    if (d <= TB) {
      if (A_ON && d <= TA) {
        sinkA(atomicAdd(cntA, 1u), i, d);
        sinkA.count1(d);
      } else {
        sinkB(atomicAdd(cntB, 1u), i, d);
        sinkB.count1(d);
      }
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
  // One thread keeps kL2Ahead bytes of the row requested ahead of the pass,
  // through the TMA engine's L2 prefetch: bytes in flight from HBM that hold
  // neither registers nor shared memory.
  constexpr uint32_t kTileBytes = G::kThreads * 32u;  // one ring step of the group
  const uint64_t body_bytes = (uint64_t)sp.nvec * 32u;
  if (tid == 0 && body_bytes > 0) {
    const uint64_t first = body_bytes < kL2Ahead ? body_bytes : kL2Ahead;
    prefetch_l2(body, (uint32_t)first);
  }
  constexpr uint32_t kSentinel = SIGNED_FAST ? 0x80000000u : 0xFFFFFFFFu;
  // Ring of kRing single-vector tiles: tile k of this thread is the vector
  // k * kThreads + rank; while tile k is filtered, tiles k+1 .. k+kRing-1 are
  // in flight.  Slot indices are compile-time (the ring is unrolled).
  const int ntiles = (sp.nvec + G::kThreads - 1) / G::kThreads;
  uint32_t buf[kRing][8];
#pragma unroll
  for (int u = 0; u < kRing - 1; ++u) {
    const int vi = u * G::kThreads + tid;
    if (vi < sp.nvec) {
      ld_stream8(body + 8 * vi, buf[u]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) buf[u][e] = kSentinel;
    }
  }
  for (int base = 0; base < ntiles; base += kRing) {
#pragma unroll
    for (int u = 0; u < kRing; ++u) {
      const int k = base + u;
      if (k >= ntiles) break;
      {
        constexpr int kAhead = kRing - 1;
        const int vp = (k + kAhead) * G::kThreads + tid;
        uint32_t* dst = buf[(u + kAhead) % kRing];
        if (vp < sp.nvec) {
          ld_stream8(body + 8 * vp, dst);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) dst[e] = kSentinel;
        }
      }
      if (tid == 0) {
        const uint64_t off = (uint64_t)k * kTileBytes + kL2Ahead;
        if (off < body_bytes) {
          const uint64_t len = body_bytes - off < kTileBytes ? body_bytes - off : kTileBytes;
          prefetch_l2(reinterpret_cast<const unsigned char*>(body) + off, (uint32_t)len);
        }
      }
      const uint32_t* x = buf[u];
      const int vi = k * G::kThreads + tid;
      bool keep;
      if (SIGNED_FAST) {
        int mx = (int)x[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) mx = max(mx, (int)x[e]);
        keep = mx >= CB;  // the sentinel is never admitted
      } else {
        uint32_t mn = desc_key(x[0]);
#pragma unroll
        for (int e = 1; e < 8; ++e) mn = min(mn, desc_key(x[e]));
        keep = vi < sp.nvec && mn <= TB;
      }
      const uint32_t bal = __ballot_sync(kFull, keep);
      if (bal != 0u) {
        if (keep) {
          const int pos = qn + __popc(bal & lt);
          uint4* qdst = reinterpret_cast<uint4*>(q.vals + 8 * pos);
          qdst[0] = make_uint4(x[0], x[1], x[2], x[3]);
          qdst[1] = make_uint4(x[4], x[5], x[6], x[7]);
          q.vidx[pos] = vi;
        }
        qn += __popc(bal);
        if (qn >= 32) {
          __syncwarp();
          drain_queue<SIGNED_FAST, A_ON>(q, qn, sp.a0, CA, CB, TA, TB, cntA, cntB, sinkA, sinkB);
          qn -= 32;
          __syncwarp();
        }
      }
    }
  }
  if (qn > 0) {
    __syncwarp();
    drain_queue<SIGNED_FAST, A_ON>(q, qn, sp.a0, CA, CB, TA, TB, cntA, cntB, sinkA, sinkB);
    __syncwarp();
  }
}

// Dispatches on the cutoff's sign (signed-compare fast path) and on whether
// class A exists.
template <class G, class SinkA, class SinkB>
__device__ __forceinline__ void scan_two_class(const float* row, int lo, int hi, uint32_t TA,
                                               uint32_t TB, bool a_on, uint32_t* cntA,
                                               uint32_t* cntB, uint32_t* queues,
                                               const SinkA& sinkA, const SinkB& sinkB) {
  const bool fast = (bits_from_desc(TB) & 0x80000000u) == 0u;
  if (fast) {
    if (a_on)
      scan_tiles<G, true, true>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
    else
      scan_tiles<G, true, false>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
  } else {
    if (a_on)
      scan_tiles<G, false, true>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
    else
      scan_tiles<G, false, false>(row, lo, hi, TA, TB, cntA, cntB, queues, sinkA, sinkB);
  }
}

// Coarse histogram over row[lo, hi) by group G (first pass of exact coarse
// recovery, eq. 20).  No group barrier.
template <class G>
__device__ void scan_coarse_hist(const float* row, int lo, int hi, uint32_t* hist) {
  if (lo >= hi) return;
  const int tid = G::rank();
  const Span sp = aligned_span(row, lo, hi);
  const int head = sp.a0 - lo, tail = hi - sp.a_end;
  if (tid < head + tail) {
    const int i = tid < head ? lo + tid : sp.a_end + (tid - head);
    atomicAdd(&hist[coarse_bin(ld_stream1(row + i))], 1u);
  }
  const float* body = row + sp.a0;
  for (int t = tid; t < sp.nvec; t += 2 * G::kThreads) {
    uint32_t x[16];
    const bool second = t + G::kThreads < sp.nvec;
    ld_stream8(body + 8 * t, x);
    if (second) ld_stream8(body + 8 * (t + G::kThreads), x + 8);
    RunHist rh;
#pragma unroll
    for (int k = 0; k < 8; ++k) rh.add(hist, (uint32_t)coarse_bin(x[k]));
    if (second) {
#pragma unroll
      for (int k = 8; k < 16; ++k) rh.add(hist, (uint32_t)coarse_bin(x[k]));
    }
    rh.flush(hist);
  }
}

// Sinks: where an admitted (position, index, key) goes.
// operator() stores one entry; count8 (the keys of u[e] for the bits e of m)
// and count1 feed the sink's histogram, if it has one.
struct NoCount {
  __device__ __forceinline__ void count8(uint32_t, const uint32_t*) const {}
  __device__ __forceinline__ void count1(uint32_t) const {}
};
struct FrontierSink : NoCount {  // frontier entry + leading-digit histogram (eqs. 17, 20)
  Frontier F;
  uint32_t* hist;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    F.put(p, i, d);
    smem_add(&hist[d >> 21], 1u);
  }
};
struct CommitSink : NoCount {  // committed straight to the output (E0 of eq. 20)
  int32_t* out_row;
  uint32_t K;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t) const {
    if (p < K) out_row[p] = i;
  }
};
struct DropSink : NoCount {
  __device__ __forceinline__ void operator()(uint32_t, int32_t, uint32_t) const {}
};

// Warp-aggregated commit of idx for the lanes where `com` holds.
__device__ __forceinline__ void commit_warp(uint32_t* n_out, int32_t* out_row, int K, bool com,
                                            int32_t idx, uint32_t lt) {
  const uint32_t bal = __ballot_sync(kFull, com);
  if (bal == 0u) return;
  uint32_t base = 0u;
  if ((threadIdx.x & 31) == 0) base = atomicAdd(n_out, (uint32_t)__popc(bal));
  base = __shfl_sync(kFull, base, 0);
  if (com) {
    const uint32_t slot = base + (uint32_t)__popc(bal & lt);
    if (slot < (uint32_t)K) out_row[slot] = idx;
  }
}

// ----------------------------------------------------------------------------
// Phase 3: prefix-commit-retain refinement (section 4.4, eqs. 22-25)
// ----------------------------------------------------------------------------

// Block-wide exclusive scan of one packed value per thread (the two 16-bit
// halves must not carry); returns this thread's exclusive prefix and the
// group total in `total`.
template <class G>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, GroupScratch& sc,
                                                         uint32_t& total) {
  const int tid = G::rank(), lane = tid & 31, warp = tid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc.warp_sums[warp] = incl;
  G::sync();
  uint32_t w = lane < G::kWarps ? sc.warp_sums[lane] : 0u;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, w, o);
    if (lane >= o) w += y;
  }
  const uint32_t before = warp ? __shfl_sync(kFull, w, warp - 1) : 0u;
  total = __shfl_sync(kFull, w, G::kWarps - 1);
  G::sync();  // warp_sums may be reused on return
  return before + incl - v;
}

// Block-wide min and max of one value per thread.
template <class G>
__device__ __forceinline__ void block_min_max(uint32_t vmin, uint32_t vmax, GroupScratch& sc,
                                              uint32_t& omin, uint32_t& omax) {
  const int tid = G::rank(), lane = tid & 31, warp = tid >> 5;
  vmin = __reduce_min_sync(kFull, vmin);
  vmax = __reduce_max_sync(kFull, vmax);
  if constexpr (G::kWarps <= 16) {
    // both partials in one round: minima in warp_sums[0, 16), maxima in [16, 32)
    if (lane == 0) {
      sc.warp_sums[warp] = vmin;
      sc.warp_sums[16 + warp] = vmax;
    }
    G::sync();
    omin = __reduce_min_sync(kFull, lane < G::kWarps ? sc.warp_sums[lane] : 0xFFFFFFFFu);
    omax = __reduce_max_sync(kFull, lane < G::kWarps ? sc.warp_sums[16 + lane] : 0u);
    G::sync();
  } else {
    if (lane == 0) sc.warp_sums[warp] = vmin;
    G::sync();
    omin = __reduce_min_sync(kFull, lane < G::kWarps ? sc.warp_sums[lane] : 0xFFFFFFFFu);
    G::sync();
    if (lane == 0) sc.warp_sums[warp] = vmax;
    G::sync();
    omax = __reduce_max_sync(kFull, lane < G::kWarps ? sc.warp_sums[lane] : 0u);
    G::sync();
  }
}

// Histogram add by a whole warp: one shared atomic when every active lane has
// the same bin (tie runs), one per lane otherwise.
__device__ __forceinline__ void hist_add_same(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t act = __ballot_sync(kFull, active);
  if (act == 0u) return;
  const int first = __ffs(act) - 1;
  const uint32_t b0 = __shfl_sync(kFull, bin, first);
  if (__ballot_sync(kFull, active && bin == b0) == act) {
    if ((int)(threadIdx.x & 31) == first) atomicAdd(&hist[b0], (uint32_t)__popc(act));
  } else if (active) {
    atomicAdd(&hist[bin], 1u);
  }
}

// The t-th smallest (1 <= t <= their count) of the values in v[0, n) that
// are <= vhi, by radix rounds of 11-bit digits taken over the values' own
// range [min, max] (so that clustered values still spread over the bins).
// Returns the value and, in `below`, how many considered values are smaller;
// `bad` when no value is considered or the counts are inconsistent.
// With `range_lo` <= every considered value (and vhi >= every one), the
// range [range_lo, vhi] is taken as given instead of measured by a pass.
template <class G>
__device__ uint32_t small_select(const uint32_t* v, uint32_t n, uint32_t vhi, uint32_t t,
                                 uint32_t* hist, GroupScratch& sc, uint32_t& below, bool& bad,
                                 bool have_range = false, uint32_t range_lo = 0u) {
  const int tid = G::rank();
  uint32_t kmin, kmax;
  if (have_range) {
    kmin = range_lo;
    kmax = vhi;
  } else {
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
    for (uint32_t i = tid; i < n; i += G::kThreads) {
      const uint32_t x = v[i];
      if (x <= vhi) {
        mn = min(mn, x);
        mx = max(mx, x);
      }
    }
    block_min_max<G>(mn, mx, sc, kmin, kmax);
  }
  below = 0u;
  bad = kmin > kmax;
  if (bad) return 0u;
  uint64_t qlo = kmin, qhi = (uint64_t)kmax + 1u;
  const uint32_t nr = (n + 31u) & ~31u;
  while (qhi - qlo > 1u) {
    const int s = 64 - __clzll((long long)(qhi - qlo - 1u));
    const int width = s < 11 ? s : 11;
    const int shift = s - width;
    const int nbins = (1 << width) < 128 ? 128 : (1 << width);
    clear_hist<G>(hist, nbins);
    G::sync();
    for (uint32_t i = tid; i < nr; i += G::kThreads) {
      const uint32_t x = i < n ? v[i] : 0xFFFFFFFFu;
      const bool in = i < n && x <= vhi && (uint64_t)x >= qlo && (uint64_t)x < qhi;
      hist_add_same(hist, in ? (uint32_t)(((uint64_t)x - qlo) >> shift) : 0u, in);
    }
    G::sync();
    find_boundaries<G>(hist, sc, nbins, 1, t, 0u);
    const int b = sc.res_bin[0];
    const uint32_t bl = sc.res_below[0], cnt = sc.res_cnt[0];
    if (b < 0) {
      bad = true;
      return 0u;
    }
    qlo += (uint64_t)b << shift;
    qhi = qlo + ((uint64_t)1 << shift);
    below += bl;
    t -= bl;
    if (cnt <= 32u && qhi - qlo > 1u) {
      // At most 32 values left in the bucket: one warp ranks them directly
      // instead of further radix rounds.
      G::sync();  // every thread has read the finder's results
      if (tid == 0) sc.bcast = 0;
      G::sync();
      uint32_t* buf = hist;  // free after the finder
      for (uint32_t i = tid; i < n; i += G::kThreads) {
        const uint32_t x = v[i];
        if (x <= vhi && (uint64_t)x >= qlo && (uint64_t)x < qhi) {
          const int slot = atomicAdd(&sc.bcast, 1);
          if (slot < 32) buf[slot] = x;
        }
      }
      G::sync();
      if (tid < 32) {
        const int m = min(sc.bcast, 32);
        const bool valid = tid < m;
        const uint32_t x = valid ? buf[tid] : 0u;
        uint32_t less = 0u, eq = 0u;
        for (int j = 0; j < 32; ++j) {
          const uint32_t y = __shfl_sync(kFull, x, j);
          if (j < m) {
            less += y < x ? 1u : 0u;
            eq += y == x ? 1u : 0u;
          }
        }
        const uint32_t hit = __ballot_sync(kFull, valid && less < t && t <= less + eq);
        const int src = hit ? __ffs(hit) - 1 : 0;
        const uint32_t vx = __shfl_sync(kFull, x, src);
        const uint32_t vl = __shfl_sync(kFull, less, src);
        if (tid == 0) {
          sc.res_bin[1] = hit ? 1 : -1;
          sc.res_cnt[1] = vx;
          sc.res_below[1] = vl;
        }
      }
      G::sync();
      if (sc.res_bin[1] < 0) {
        bad = true;
        return 0u;
      }
      below += sc.res_below[1];
      return sc.res_cnt[1];
    }
  }
  return (uint32_t)qlo;
}


// Phase 3 (eqs. 22-25) with the commits of every digit deferred to one final
// pass.  Round j only needs h_j over the frontier entries whose leading digits
// match b_0..b_{j-1} (Q_j) to find b_j = min{b : H_j(b) >= k_j} and k_{j+1} =
// k_j - H_j(b_j - 1); the union of the groups R_j committed per round is
// exactly {key < T*} with T* the key spelled by (b_0, b_1, b_2), and Q_3 is
// {key == T*}, from which k_3 entries fill the rest.  When H_j(b_j) == k_j the
// boundary group closes the quota at round j and no tie fill is needed.  The
// frontier is only read (shared memory or its global slice), never moved.
// Entry: frontier holds n entries (Q0), hist holds h0, k = k0 indices remain,
// sl.n_out = |E0|.  Exit: sl.n_out == K.
//
// When round 0 leaves the quota open on a frontier that spilled out of shared
// memory (tie runs, constant rows), the keys of Q_1 (at most `scap`) are
// compacted into `scratch` and the remaining digits are resolved there with
// small_select: the same threshold, reached without further passes over the
// global slice.
template <class G>
__device__ void refine_digits(const Frontier& F, uint32_t n, uint32_t k, uint32_t* hist,
                              GroupScratch& sc, Slot& sl, int32_t* out_row, int K,
                              uint32_t* scratch, uint32_t scap) {
  const int tid = G::rank();
  const uint32_t lt = lanemask_lt();
  const uint32_t nr = (n + 31u) & ~31u;  // whole warps visit every slot index
  uint64_t commit_below = 0;             // commit keys < commit_below
  uint32_t tie_key = 0u, ties = 0u;      // then `ties` entries with key == tie_key
  uint32_t prefix = 0u;                  // b_0 .. b_{j-1}
  bool resolved = false;
  for (int j = 0; j < 3 && k > 0; ++j) {
    const int width = j == 2 ? 10 : 11;
    const int shift = j == 0 ? 21 : (j == 1 ? 10 : 0);  // digit j occupies bits [shift, shift+width)
    find_boundaries<G>(hist, sc, 1 << width, 1, k, 0u);
    const int b = sc.res_bin[0];
    const uint32_t below = sc.res_below[0], cnt = sc.res_cnt[0];
    if (b < 0) {  // inconsistent counts: cannot happen; finish_row flags it
      k = 0;
      resolved = true;
      break;
    }
    prefix = (prefix << width) | (uint32_t)b;
    if (below + cnt == k) {
      // Bucket b_j closes the quota: commit every key whose leading digits
      // are <= (b_0 .. b_j).
      commit_below = (uint64_t)(prefix + 1u) << shift;
      k = 0;
      resolved = true;
      break;
    }
    k -= below;
    if (j == 0 && cnt <= scap && n > F.cap) {
      // Q_1 = frontier keys whose digit 0 is b_0: compact them, then select
      // the k-th smallest among them.
      G::sync();  // every thread has read the finder's results
      if (tid == 0) sc.bcast = 0;
      G::sync();
      for (uint32_t p0 = 0; p0 < nr; p0 += kRefineBatch * G::kThreads) {
        uint32_t d[kRefineBatch];
#pragma unroll
        for (int bb = 0; bb < kRefineBatch; ++bb) {
          const uint32_t pp = p0 + bb * G::kThreads + tid;
          int32_t i;
          d[bb] = 0xFFFFFFFFu;
          if (pp < n) F.get(pp, i, d[bb]);
        }
#pragma unroll
        for (int bb = 0; bb < kRefineBatch; ++bb) {
          const uint32_t pp = p0 + bb * G::kThreads + tid;
          if (p0 + bb * G::kThreads >= nr) break;  // warp-uniform
          const bool in = pp < n && (d[bb] >> 21) == prefix;
          const uint32_t bal = __ballot_sync(kFull, in);
          if (bal != 0u) {
            uint32_t base = 0u;
            if ((tid & 31) == 0) base = (uint32_t)atomicAdd(&sc.bcast, __popc(bal));
            base = __shfl_sync(kFull, base, 0);
            const uint32_t slot = base + (uint32_t)__popc(bal & lt);
            if (in && slot < scap) scratch[slot] = d[bb];
          }
        }
      }
      G::sync();
      uint32_t below1;
      bool bad = false;
      const uint32_t vstar = small_select<G>(scratch, cnt, 0xFFFFFFFFu, k, hist, sc, below1, bad);
      if (bad) {  // inconsistent counts: cannot happen; finish_row flags it
        k = 0;
        resolved = true;
        break;
      }
      commit_below = vstar;
      tie_key = vstar;
      ties = k - below1;
      resolved = true;
      break;
    }
    if (j == 2) {
      commit_below = prefix;  // the full key T*
      tie_key = prefix;
      ties = k;
      resolved = true;
      break;
    }
    // h_{j+1} over Q_{j+1} = entries whose digits 0..j equal prefix.
    G::sync();  // the finder is done with hist
    clear_hist<G>(hist, 2048);
    G::sync();
    // Eight entries per thread in flight (the frontier may live in global
    // memory), then run-length merged histogram adds.
    for (uint32_t p0 = 0; p0 < n; p0 += kRefineBatch * G::kThreads) {
      uint32_t d[kRefineBatch];
#pragma unroll
      for (int b = 0; b < kRefineBatch; ++b) {
        const uint32_t pp = p0 + b * G::kThreads + tid;
        int32_t i;
        d[b] = 0xFFFFFFFFu;
        if (pp < n) F.get(pp, i, d[b]);
      }
      RunHist rh;
#pragma unroll
      for (int b = 0; b < kRefineBatch; ++b) {
        const uint32_t pp = p0 + b * G::kThreads + tid;
        if (pp < n && (d[b] >> shift) == prefix) rh.add(hist, digit(d[b], j + 1));
      }
      rh.flush(hist);
    }
    G::sync();
  }
  if (resolved) {
    if (tid == 0) sl.n_keep = 0u;
    G::sync();
    for (uint32_t p0 = 0; p0 < nr; p0 += kCommitBatch * G::kThreads) {
      int32_t ib[kCommitBatch];
      uint32_t db[kCommitBatch];
#pragma unroll
      for (int b = 0; b < kCommitBatch; ++b) {
        const uint32_t pp = p0 + b * G::kThreads + tid;
        ib[b] = -1;
        db[b] = 0xFFFFFFFFu;
        if (pp < n) F.get(pp, ib[b], db[b]);
      }
#pragma unroll
      for (int b = 0; b < kCommitBatch; ++b) {
        const uint32_t pp = p0 + b * G::kThreads + tid;
        if (p0 + b * G::kThreads >= nr) break;  // warp-uniform: nr and the stride are multiples of 32
        const bool in = pp < n;
        const uint32_t d = db[b];
        const bool com = in && (uint64_t)d < commit_below;
        const bool tie = in && ties > 0u && d == tie_key;
        const uint32_t tb = __ballot_sync(kFull, tie);
        bool take = false;
        if (tb) {
          uint32_t base = 0u;
          if ((threadIdx.x & 31) == 0) base = atomicAdd(&sl.n_keep, (uint32_t)__popc(tb));
          base = __shfl_sync(kFull, base, 0);
          take = tie && base + (uint32_t)__popc(tb & lt) < ties;
        }
        commit_warp(&sl.n_out, out_row, K, com || take, ib[b], lt);
      }
    }
  }
  G::sync();
}

// h0 of eq. 17 (leading 11-bit digit of every frontier key) rebuilt from a
// frontier held in shared memory.
template <class G>
__device__ void rebuild_h0(const Frontier& F, uint32_t n, uint32_t* hist) {
  G::sync();
  clear_hist<G>(hist, 2048);
  G::sync();
  for (uint32_t p = G::rank(); p < n; p += G::kThreads) smem_add(&hist[F.s[p].y >> 21], 1u);
  G::sync();
}

// Phase 3 for a frontier held in shared memory (n <= F.cap), reaching the
// same threshold as eqs. 22-25 with digits taken over the frontier's own key
// range [kmin, kmax] instead of fixed bit fields: frontier keys cluster in a
// few leading-digit buckets, so a range-relative 11-bit digit usually leaves
// a boundary bucket of a handful of keys after one histogram.  One pass then
// commits every key below the boundary bucket and collects that bucket, whose
// k' smallest keys are taken by one warp (32 keys or fewer) or by
// small_select.  A frontier whose keys are all equal commits any k of them
// (the tie fill of eq. 25).  Returns false, with nothing committed and h0
// restored in `hist`, when the boundary bucket outgrows `scratch` (pcap
// (key, index) pairs: keys at [0, pcap), indices at [pcap, 2 pcap)); the
// caller then runs the fixed-digit recurrence.
template <class G>
__device__ bool refine_fast(const Frontier& F, uint32_t n, uint32_t k, uint32_t* hist,
                            GroupScratch& sc, Slot& sl, int32_t* out_row, int K,
                            uint32_t* scratch, uint32_t pcap) {
  const int tid = G::rank();
  const uint32_t lt = lanemask_lt();
  const uint32_t nr = (n + 31u) & ~31u;
  if (k == 0u || n < k) return k == 0u;  // n < k: inconsistent counts; finish_row flags it
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (uint32_t p = tid; p < n; p += G::kThreads) {
    const uint32_t d = F.s[p].y;
    mn = min(mn, d);
    mx = max(mx, d);
  }
  uint32_t kmin, kmax;
  block_min_max<G>(mn, mx, sc, kmin, kmax);
  if (kmin == kmax) {
    // every frontier key is equal: any k entries complete the selection
    const uint32_t base = sl.n_out;
    for (uint32_t p = tid; p < k; p += G::kThreads)
      if (base + p < (uint32_t)K) out_row[base + p] = (int32_t)F.s[p].x;
    G::sync();
    if (tid == 0) sl.n_out = base + k;
    G::sync();
    return true;
  }
  const uint32_t range = kmax - kmin;
  const int width = 32 - __clz((int)range);  // bits of the range (range >= 1)
  const int shift = width > 11 ? width - 11 : 0;
  const int nbins = (int)(((range >> shift) + 1u + 127u) & ~127u);  // <= 2048
  clear_hist<G>(hist, nbins);
  G::sync();
  for (uint32_t p = tid; p < n; p += G::kThreads)
    smem_add(&hist[(F.s[p].y - kmin) >> shift], 1u);
  G::sync();
  find_boundaries<G>(hist, sc, nbins, 1, k, 0u);
  const int b = sc.res_bin[0];
  const uint32_t below = sc.res_below[0], cnt = sc.res_cnt[0];
  const uint32_t kk = k - below;  // keys still wanted from bucket b (1 <= kk <= cnt)
  const bool whole = b >= 0 && kk == cnt;
  if (b < 0 || (!whole && cnt > pcap)) {
    rebuild_h0<G>(F, n, hist);
    return false;
  }
  if (tid == 0) sc.bcast = 0;
  G::sync();
  uint32_t* ckey = scratch;
  int32_t* cidx = reinterpret_cast<int32_t*>(scratch + pcap);
  for (uint32_t p0 = 0; p0 < nr; p0 += G::kThreads) {
    const uint32_t p = p0 + tid;
    const bool in = p < n;
    uint2 e = make_uint2(0u, 0xFFFFFFFFu);
    if (in) e = F.s[p];
    const uint32_t bin = (e.y - kmin) >> shift;
    const bool com = in && (bin < (uint32_t)b || (whole && bin == (uint32_t)b));
    commit_warp(&sl.n_out, out_row, K, com, (int32_t)e.x, lt);
    if (!whole) {
      const bool col = in && bin == (uint32_t)b;
      const uint32_t bal = __ballot_sync(kFull, col);
      if (bal != 0u) {
        uint32_t base = 0u;
        if ((tid & 31) == 0) base = (uint32_t)atomicAdd(&sc.bcast, __popc(bal));
        base = __shfl_sync(kFull, base, 0);
        if (col) {
          const uint32_t slot = base + (uint32_t)__popc(bal & lt);
          ckey[slot] = e.y;
          cidx[slot] = (int32_t)e.x;
        }
      }
    }
  }
  G::sync();
  if (whole) return true;
  if (cnt <= 32u) {
    // One warp ranks the bucket: a key's rank counts the smaller keys and
    // the equal keys in lower lanes, so exactly kk lanes take.
    if (tid < 32) {
      const bool valid = (uint32_t)tid < cnt;
      const uint32_t x = valid ? ckey[tid] : 0xFFFFFFFFu;
      const int32_t xi = valid ? cidx[tid] : -1;
      uint32_t rank = 0u;
      for (int j = 0; j < 32; ++j) {
        const uint32_t y = __shfl_sync(kFull, x, j);
        if ((uint32_t)j < cnt && (y < x || (y == x && j < tid))) ++rank;
      }
      commit_warp(&sl.n_out, out_row, K, valid && rank < kk, xi, lt);
    }
    G::sync();
    return true;
  }
  uint32_t below1;
  bool bad = false;
  const uint32_t vstar = small_select<G>(ckey, cnt, 0xFFFFFFFFu, kk, hist, sc, below1, bad);
  if (bad) {  // inconsistent counts: cannot happen; finish_row flags it
    G::sync();
    return true;
  }
  const uint32_t ties = kk - below1;
  if (tid == 0) sl.n_keep = 0u;
  G::sync();
  const uint32_t cr = (cnt + 31u) & ~31u;
  for (uint32_t p0 = 0; p0 < cr; p0 += G::kThreads) {
    const uint32_t p = p0 + tid;
    const bool in = p < cnt;
    const uint32_t d = in ? ckey[p] : 0xFFFFFFFFu;
    const bool com = in && d < vstar;
    const bool tie = in && d == vstar;
    const uint32_t tb = __ballot_sync(kFull, tie);
    bool take = false;
    if (tb) {
      uint32_t base = 0u;
      if ((tid & 31) == 0) base = atomicAdd(&sl.n_keep, (uint32_t)__popc(tb));
      base = __shfl_sync(kFull, base, 0);
      take = tie && base + (uint32_t)__popc(tb & lt) < ties;
    }
    commit_warp(&sl.n_out, out_row, K, com || take, in ? cidx[p] : -1, lt);
  }
  G::sync();
  return true;
}

// Phase 3 of a row: the range-relative form above when the frontier is in
// shared memory and its boundary bucket fits `scratch` (scap words), the
// fixed 11+11+10 digits of eqs. 22-25 otherwise.
template <class G>
__device__ void refine(const Frontier& F, uint32_t n, uint32_t k, uint32_t* hist,
                       GroupScratch& sc, Slot& sl, int32_t* out_row, int K, uint32_t* scratch,
                       uint32_t scap) {
  if (n <= F.cap && refine_fast<G>(F, n, k, hist, sc, sl, out_row, K, scratch, scap / 2u))
    return;
  refine_digits<G>(F, n, k, hist, sc, sl, out_row, K, scratch, scap);
}

// ----------------------------------------------------------------------------
// Phase 3 over the row itself (frontiers too large to hold)
// ----------------------------------------------------------------------------

// Over the keys d <= T in [qlo, qhi) of row[0, L), by group G: each thread's
// count, smallest and largest key and how many keys equal each (accumulated
// into cnt, mn, mx, nmn, nmx), and, when `hist` is not null, the histogram of
// the digits (d - hlo) >> shift of those at or above hlo, with their count in
// nh.  Two 256-bit loads per thread in flight; a thread's adds merge runs of
// one digit across the whole pass.  No group barrier.
template <class G>
__device__ void scan_key_hist(const float* row, int L, uint32_t T, uint64_t qlo, uint64_t qhi,
                              uint64_t hlo, int shift, uint32_t* hist, uint32_t& cnt,
                              uint32_t& mn, uint32_t& mx, uint32_t& nmn, uint32_t& nmx,
                              uint32_t& nh) {
  const int tid = G::rank();
  const Span sp = aligned_span(row, 0, L);
  // keys in play: lo <= d <= hi, one unsigned offset compare; histogrammed:
  // hl <= d <= hi
  const uint64_t top = qhi == 0u ? 0u : (qhi - 1u < (uint64_t)T ? qhi - 1u : (uint64_t)T);
  if (qhi == 0u || qlo > top) return;
  const uint32_t lo = (uint32_t)qlo, span = (uint32_t)(top - qlo);
  const bool hon = hist != nullptr && hlo <= top;
  const uint32_t hl = (uint32_t)(hlo > qlo ? hlo : qlo), hspan = hon ? (uint32_t)(top - hl) : 0u;
  RunHist rh;
  auto take = [&](uint32_t d) {
    if (d - lo <= span) {
      ++cnt;
      if (d <= mn) {
        nmn = d == mn ? nmn + 1u : 1u;
        mn = d;
      }
      if (d >= mx) {
        nmx = d == mx ? nmx + 1u : 1u;
        mx = d;
      }
      const uint32_t h = d - hl;
      if (hon && h <= hspan) {
        ++nh;
        rh.add(hist, h >> shift);
      }
    }
  };
  const int head = sp.a0, tail = L - sp.a_end;
  if (tid < head + tail)
    take(desc_key(ld_stream1(row + (tid < head ? tid : sp.a_end + (tid - head)))));
  const float* body = row + sp.a0;
  constexpr int kV = 2;
  for (int t0 = 0; t0 < sp.nvec; t0 += kV * G::kThreads) {
    uint32_t x[kV][8];
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int v = t0 + k * G::kThreads + tid;
      if (v < sp.nvec) {
        ld_stream8(body + 8 * v, x[k]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[k][e] = 0xFFFFFFFFu;
      }
    }
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      if (t0 + k * G::kThreads + tid >= sp.nvec) break;
#pragma unroll
      for (int e = 0; e < 8; ++e) take(desc_key(x[k][e]));
    }
  }
  if (hon) rh.flush(hist);
}

// Visits row[0, L) by group G one 8-score vector per thread and step, two
// vectors per thread in flight: step(x, i0, nvalid) gets the bit patterns of
// positions i0 .. i0 + nvalid - 1 (whole warps call it together; the
// unaligned head and tail come first, one score per lane of warp 0).  Before
// each step of two vectors the warp asks stop() (warp-uniform) whether the
// rest of the row can be skipped.  No group barrier.
template <class G, class Step, class Stop>
__device__ __forceinline__ void visit_row(const float* row, int L, const Step& step,
                                          const Stop& stop) {
  const int tid = G::rank();
  const Span sp = aligned_span(row, 0, L);
  const int head = sp.a0, tail = L - sp.a_end;
  if (tid < 32) {  // the scalar head and tail (at most 14 scores), one lane each
    uint32_t x[8];
    const bool valid = tid < head + tail;
    const int i = tid < head ? tid : sp.a_end + (tid - head);
    x[0] = valid ? ld_stream1(row + i) : 0xFFFFFFFFu;
#pragma unroll
    for (int e = 1; e < 8; ++e) x[e] = 0xFFFFFFFFu;
    step(x, i, valid ? 1 : 0);
  }
  const float* body = row + sp.a0;
  constexpr int kV = 2;  // vectors per thread in flight
  const int nvr = (sp.nvec + 31) & ~31;
  for (int t0 = 0; t0 < nvr; t0 += kV * G::kThreads) {
    if (t0 + 32 * (tid >> 5) >= nvr || stop()) break;  // warp-uniform
    uint32_t x[kV][8];
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int v = t0 + k * G::kThreads + tid;
      if (v < sp.nvec) {
        ld_stream8(body + 8 * v, x[k]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[k][e] = 0xFFFFFFFFu;
      }
    }
#pragma unroll
    for (int k = 0; k < kV; ++k) {
      const int v = t0 + k * G::kThreads + tid;
      if (t0 + k * G::kThreads + 32 * (tid >> 5) >= nvr) break;  // warp-uniform
      step(x[k], sp.a0 + 8 * v, v < sp.nvec ? 8 : 0);
    }
  }
}

// Exclusive warp scan of v; `total` gets the warp's sum.
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, uint32_t& total) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  total = __shfl_sync(kFull, incl, 31);
  return incl - v;
}

// Places the positions i0 + e (bits e of m) at consecutive output slots from
// the warp's share of *n_out (one atomic per warp); slots >= K are dropped.
__device__ __forceinline__ void commit_mask(uint32_t m, int i0, uint32_t* n_out, int32_t* out_row,
                                            int K) {
  uint32_t tot;
  const uint32_t ex = warp_excl_scan((uint32_t)__popc(m), tot);
  if (tot == 0u) return;
  uint32_t base = 0u;
  if ((threadIdx.x & 31) == 0) base = atomicAdd(n_out, tot);
  uint32_t slot = __shfl_sync(kFull, base, 0) + ex;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (m & (1u << e)) {
      if (slot < (uint32_t)K) out_row[slot] = i0 + e;
      ++slot;
    }
  }
}

// Commit pass over row[0, L) by group G: every key d <= T in [commit_lo,
// commit_below) goes to the output, then the first `ties` keys equal to
// tie_key (ranked through sl.n_keep).  Per thread and 8-score vector, the
// committed and tied positions are bit masks; one warp scan ranks the ties
// and one places the outputs.  The pass ends as soon as all K output slots
// are taken (a row of ties stops after its first K).  Ends with a group
// barrier.
template <class G>
__device__ void scan_commit(const float* row, int L, uint32_t T, uint64_t commit_lo,
                            uint64_t commit_below, uint32_t tie_key, uint32_t ties, Slot& sl,
                            int32_t* out_row, int K) {
  if (G::rank() == 0) {
    sl.n_keep = 0u;
    prefetch_row_l2(row, L);
  }
  G::sync();
  auto step = [&](const uint32_t* x, int i0, int nvalid) {
    uint32_t cm = 0u, tm = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t d = desc_key(x[e]);
      const bool ok = e < nvalid && d <= T;
      if (ok && (uint64_t)d >= commit_lo && (uint64_t)d < commit_below)
        cm |= 1u << e;
      else if (ok && ties > 0u && d == tie_key)
        tm |= 1u << e;
    }
    if (tm != 0u && *(volatile uint32_t*)&sl.n_keep >= ties) tm = 0u;  // ties complete
    if (__ballot_sync(kFull, (cm | tm) != 0u) == 0u) return;
    if (__ballot_sync(kFull, tm != 0u) != 0u) {
      uint32_t tt;
      const uint32_t tex = warp_excl_scan((uint32_t)__popc(tm), tt);
      uint32_t base = 0u;
      if ((threadIdx.x & 31) == 0) base = atomicAdd(&sl.n_keep, tt);
      // keep the ties ranked below `ties`
      uint32_t rank = __shfl_sync(kFull, base, 0) + tex;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (tm & (1u << e)) {
          if (rank >= ties) tm &= ~(1u << e);
          ++rank;
        }
      }
    }
    commit_mask(cm | tm, i0, &sl.n_out, out_row, K);
  };
  auto full = [&]() {
    return __shfl_sync(kFull, *(volatile uint32_t*)&sl.n_out, 0) >= (uint32_t)K;
  };
  visit_row<G>(row, L, step, full);
  G::sync();
}

// ----------------------------------------------------------------------------
// Row-level building blocks
// ----------------------------------------------------------------------------

template <class G>
__device__ void write_pad_row(int32_t* out_row, int L, int K) {
  for (int t = G::rank(); t < K; t += G::kThreads) out_row[t] = t < L ? t : -1;
}

// Route record of a row (written by one thread).
__device__ __forceinline__ void write_trace(const Params& p, int row, int route, int tau0, int tau1,
                                            int c0, int c1, int tstar, int e0, int q0) {
  if (p.trace == nullptr) return;
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

__device__ __forceinline__ void write_slot_trace(const Params& p, const Slot& sl) {
  write_trace(p, sl.row, sl.route, sl.tau0, sl.tau1, sl.c0, sl.c1, sl.tstar, sl.e0, sl.q0n);
}

// Final guard: every output slot must be written exactly once.
template <class G>
__device__ void finish_row(const Params& p, Slot& sl, int32_t* out_row) {
  G::sync();
  const uint32_t used = sl.n_out;
  if (used != (uint32_t)p.K) {
    for (uint32_t t = used + G::rank(); t < (uint32_t)p.K; t += G::kThreads) out_row[t] = -1;
    if (G::rank() == 0) flag_status(p.counters, 1);
  }
  G::sync();
}

// Cutoffs of the exact coarse boundary tau* (group warps 0 and 1):
// T1 admits c <= tau*, T0 admits c < tau* (none when tau* == 0).
template <class G>
__device__ void exact_cutoffs(Slot& sl, int tstar) {
  const int warp = G::rank() >> 5;
  if (warp == 0) {
    const uint32_t t = cutoff_fast_warp(tstar);
    if ((G::rank() & 31) == 0) sl.T1 = t;
  } else if (warp == 1) {
    const uint32_t t = tstar > 0 ? cutoff_fast_warp(tstar - 1) : 0u;
    if ((G::rank() & 31) == 0) sl.T0 = t;
  }
  G::sync();
}

// Exact coarse recovery over row[0, L) (eq. 20): coarse histogram, tau* =
// min{b : C(b) >= K}, then one pass that commits c < tau* to the output (E0)
// and keeps c == tau* as the frontier Q0 with its digit-0 histogram h0.
// Leaves the refinement interface in the slot: n_front = |Q0|, n_out = |E0|.
template <class G>
__device__ void exact_recovery(const Params& p, const float* row, int L, const Frontier& F,
                               uint32_t* hist, GroupScratch& sc, Slot& sl, int32_t* out_row,
                               uint32_t* queues) {
  const int K = p.K;
  clear_hist<G>(hist, 2048);
  if (G::rank() == 0) {
    sl.n_front = 0u;
    sl.n_out = 0u;
  }
  G::sync();
  scan_coarse_hist<G>(row, 0, L, hist);
  G::sync();
  find_boundaries<G>(hist, sc, 2048, 1, (uint32_t)K, 0u);
  const int tstar = sc.res_bin[0];
  const int e0 = (int)sc.res_below[0];
  exact_cutoffs<G>(sl, tstar);
  const uint32_t tlo = sl.T0, thi = sl.T1;
  clear_hist<G>(hist, 2048);
  G::sync();
  CommitSink commit_sink{{}, out_row, (uint32_t)K};
  FrontierSink front_sink{{}, F, hist};
  scan_two_class<G>(row, 0, L, tlo, thi, tstar > 0, &sl.n_out, &sl.n_front, queues, commit_sink,
                    front_sink);
  G::sync();
  if (G::rank() == 0) {
    sl.tstar = tstar;
    sl.e0 = e0;
    sl.q0n = (int)sl.n_front;
  }
  G::sync();
}

// Exact coarse recovery bounded by the view (sampled rows).  Phase 2 left
// cb < K keys in the frontier, every key d <= Tb (the cutoff of bin tau_b),
// so the K-th key lies in a later coarse bin.  The view's histogram predicts
// how many keys the next bins hold: one pass appends Tb < d <= T2, T2 the
// cutoff of the first bin b2 (at most 32 bins on) whose predicted addition
// covers twice the shortfall plus two view strides.  When the frontier then
// holds K keys or more, it holds every key of the bins up to b2, so its
// coarse histogram gives tau*, |E0| and |Q0| of eq. 20 exactly, and it holds
// the whole Top-K: Phase 3 refines it with k = K and nothing committed.  The
// result is that of the full-row recovery with one pass over the row instead
// of two (a full-row coarse histogram is one shared-memory add per score).
// Returns false when no bin qualifies or the count still falls short; the
// caller then runs the full-row recovery.  `view` holds the row's view
// histogram on entry and the frontier's coarse histogram on a true return.
template <class G>
__device__ bool bounded_recovery(const Params& p, const float* row, int L, const Frontier& F,
                                 uint32_t* hist, uint32_t* view, GroupScratch& sc, Slot& sl,
                                 uint32_t* queues, uint32_t Tb, int tau_b) {
  const uint32_t K = (uint32_t)p.K;
  if (G::rank() < 32) {
    const int lane = G::rank();
    const int b = tau_b + 1 + lane;
    uint32_t v = b < kCoarseBins ? view[b] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += t;
    }
    const uint64_t need = 2ull * (K - sl.n_front) + 2ull * (uint32_t)p.s;
    const unsigned m =
        __ballot_sync(kFull, b < kCoarseBins && (uint64_t)v * (uint32_t)p.s >= need);
    const int b2 = m != 0u ? tau_b + __ffs((int)m) : -1;  // first qualifying bin
    uint32_t T2 = 0u;
    if (b2 >= 0) T2 = cutoff_fast_warp(b2);
    if (lane == 0) {
      sc.bcast = b2;
      sc.bcast2 = (int32_t)T2;
    }
  }
  G::sync();
  const int b2 = sc.bcast;
  const uint32_t T2 = (uint32_t)sc.bcast2;
  if (b2 < 0) return false;
  FrontierSink front_sink{{}, F, hist};
  DropSink drop;
  scan_two_class<G>(row, 0, L, Tb, T2, true, &sl.n_drop, &sl.n_front, queues, drop, front_sink);
  G::sync();
  const uint32_t c2 = sl.n_front;
  if (c2 < K) return false;
  clear_hist<G>(view, kCoarseBins);
  G::sync();
  for (uint32_t q = G::rank(); q < c2; q += G::kThreads) {
    int32_t i;
    uint32_t d;
    F.get(q, i, d);
    smem_add(&view[coarse_bin(bits_from_desc(d), d)], 1u);
  }
  G::sync();
  find_boundaries<G>(view, sc, kCoarseBins, 1, K, 0u);
  if (G::rank() == 0) {
    sl.tstar = sc.res_bin[0];
    sl.e0 = (int32_t)sc.res_below[0];
    sl.q0n = (int32_t)sc.res_cnt[0];
  }
  G::sync();
  return true;
}

// Exact coarse recovery with the row resident in registers (section 5.5,
// "Row-local exact": the short-row specialization keeps aligned score vectors
// in registers across boundary construction and classification).
template <class G, int VPT>
__device__ void exact_recovery_resident(const Params& p, const float* row, int L,
                                        const Frontier& F, uint32_t* hist, GroupScratch& sc,
                                        Slot& sl, int32_t* out_row) {
  const int K = p.K;
  const int tid = G::rank();
  const uint32_t lt = lanemask_lt();
  uint32_t v[VPT];
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 31u) == 0u;
#pragma unroll
  for (int g = 0; g < VPT / 8; ++g) {
    const int i0 = (g * G::kThreads + tid) * 8;
    if (aligned && i0 + 7 < L) {
      ld_stream8(row + i0, v + 8 * g);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[g * 8 + e] = (i0 + e < L) ? ld_stream1(row + i0 + e) : 0u;
    }
  }
  clear_hist<G>(hist, 2048);
  if (tid == 0) {
    sl.n_front = 0u;
    sl.n_out = 0u;
  }
  G::sync();
  {
    RunHist rh;
#pragma unroll
    for (int g = 0; g < VPT / 8; ++g) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = (g * G::kThreads + tid) * 8 + e;
        if (i < L) rh.add(hist, (uint32_t)coarse_bin(v[g * 8 + e]));
      }
    }
    rh.flush(hist);
  }
  G::sync();
  find_boundaries<G>(hist, sc, 2048, 1, (uint32_t)K, 0u);
  const int tstar = sc.res_bin[0];
  const int e0 = (int)sc.res_below[0];
  exact_cutoffs<G>(sl, tstar);
  clear_hist<G>(hist, 2048);
  G::sync();
  const uint32_t tlo = sl.T0, thi = sl.T1;
  const bool has_lo = tstar > 0;
#pragma unroll
  for (int g = 0; g < VPT / 8; ++g) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = (g * G::kThreads + tid) * 8 + e;
      const uint32_t d = desc_key(v[g * 8 + e]);
      const bool valid = i < L && d <= thi;
      const bool com = valid && has_lo && d <= tlo;
      commit_warp(&sl.n_out, out_row, K, com, i, lt);
      const bool keep = valid && !com;
      const uint32_t kb = __ballot_sync(kFull, keep);
      if (kb != 0u) {
        uint32_t base = 0u;
        if ((tid & 31) == 0) base = atomicAdd(&sl.n_front, (uint32_t)__popc(kb));
        base = __shfl_sync(kFull, base, 0);
        if (keep) {
          F.put(base + (uint32_t)__popc(kb & lt), i, d);
          atomicAdd(&hist[d >> 21], 1u);
        }
      }
    }
  }
  G::sync();
  if (tid == 0) {
    sl.tstar = tstar;
    sl.e0 = e0;
    sl.q0n = (int)sl.n_front;
  }
  G::sync();
}

__device__ __forceinline__ int view_phase(int row, int s, int s_bits) {
  if (s_bits == 0) return 0;
  return (int)(__brev((uint32_t)(row & (s - 1))) >> (32 - s_bits));
}

__device__ __forceinline__ int view_size(int L, int a, int s) {
  return L > a ? (L - a + s - 1) / s : 0;
}

// Boundaries tau0 / tau1 of a complete view histogram (eq. 15: the first bins
// whose inclusive prefix reaches q0 / q1) and their inclusive cutoffs (section
// 4.3), written to the slot.
template <class G>
__device__ void view_cutoffs(const Params& p, const uint32_t* hist, GroupScratch& sc, Slot& sl) {
  find_boundaries<G>(hist, sc, 2048, p.dual ? 2 : 1, (uint32_t)p.q0, (uint32_t)p.q1);
  const int warp = G::rank() >> 5;
  if (warp == 0 || (warp == 1 && p.dual)) {
    const int b = sc.res_bin[warp];
    const uint32_t t = cutoff_fast_warp(b);
    if ((G::rank() & 31) == 0) {
      if (warp == 0) {
        sl.T0 = t;
        sl.tau0 = b;
        sl.vcnt0 = b >= 0 ? sc.res_below[0] + sc.res_cnt[0] : 0u;
      } else {
        sl.T1 = t;
        sl.tau1 = b;
        sl.vcnt1 = b >= 0 ? sc.res_below[1] + sc.res_cnt[1] : 0u;
      }
    }
  } else if (warp == 1 && G::rank() == 32) {
    sl.T1 = 0u;
    sl.tau1 = -1;
    sl.vcnt1 = 0u;
  }
  G::sync();
}

// Phase 1 (section 4.2, eqs. 13-15) by group G: coarse histogram of the view
// V = {i < L : i = a_r (mod s)}, the boundaries tau0 / tau1 and their
// inclusive cutoffs, written to the slot.  Each thread issues up to 8 view
// loads before using any.  Entered with a cleared histogram; leaves it dirty.
template <class G>
__device__ void sample_view(const Params& p, const float* row, int L, int a, uint32_t* hist,
                            GroupScratch& sc, Slot& sl) {
  const int nv = view_size(L, a, p.s);
  const int tid = G::rank();
  for (int t0 = 0; t0 < nv; t0 += 8 * G::kThreads) {
    uint32_t u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int t = t0 + k * G::kThreads + tid;
      u[k] = t < nv ? __ldg(reinterpret_cast<const unsigned int*>(row) + a + (int64_t)t * p.s) : 0u;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (t0 + k * G::kThreads + tid < nv) smem_add(&hist[coarse_bin(u[k])], 1u);
  }
  G::sync();
  view_cutoffs<G>(p, hist, sc, sl);
}

// Optional guess source (previous-step Top-K): the worst coarse bin of the K
// guessed scores, valid only when all K entries are positions of this row.
// On success the slot holds tau0 = that bin and T0 = its cutoff.
template <class G>
__device__ bool guess_bin(const Params& p, const float* row, int L, int r, GroupScratch& sc,
                          Slot& sl) {
  if (G::rank() == 0) {
    sc.gmax = -1;
    sc.ginvalid = 0;
  }
  G::sync();
  const int32_t* g = p.prev + (int64_t)r * p.K;
  int worst = -1, invalid = 0;
  for (int t = G::rank(); t < p.K; t += G::kThreads) {
    const int32_t idx = g[t];
    if (idx < 0 || idx >= L) {
      invalid = 1;
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(row) + idx);
      worst = max(worst, coarse_bin(u));
    }
  }
  if (invalid) atomicOr(&sc.ginvalid, 1);
  if (worst >= 0) atomicMax(&sc.gmax, worst);
  G::sync();
  const bool ok = sc.ginvalid == 0;
  if (ok && G::rank() < 32) {
    const uint32_t t = cutoff_fast_warp(sc.gmax);
    if (G::rank() == 0) {
      sl.T0 = t;
      sl.tau0 = sc.gmax;
    }
  }
  G::sync();
  return ok;
}

__device__ __forceinline__ int live_rows(const Params& p) {
  int m = p.num_valid_rows ? *p.num_valid_rows : p.M_cap;
  return m < 0 ? 0 : (m > p.M_cap ? p.M_cap : m);
}

__device__ __forceinline__ int row_length(const Params& p, int r) {
  const int L = p.ke[r];
  return L < 0 ? 0 : (L > p.N ? p.N : L);
}

__device__ __forceinline__ Frontier make_frontier(const Params& p, uint2* smem_part,
                                                  int64_t slice) {
  Frontier F;
  F.s = smem_part;
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

// Last CTA out resets the queue head and the exit counter (section 5.5:
// "persistent counters are restored on device").  Entered by the whole CTA.
__device__ void exit_protocol(int32_t* counters) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(counters + kCtrExit, 1);
    if (prev == (int)(gridDim.x * gridDim.y) - 1) {
      atomicExch(counters + kCtrQueue, 0);
      atomicExch(counters + kCtrExit, 0);
      atomicExch(counters + kCtrDeferred, 0);
    }
  }
}

// ----------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and TMA copies
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One TMA bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Bounded wait for phase 0 of `bar`; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar) {
  for (int it = 0; it < (1 << 20); ++it)
    if (mbar_try_wait(bar, 0u)) return true;
  return false;
}

// Bounded wait for phase `parity` of `bar`; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_parity_bounded(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < (1 << 20); ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// One tiled TMA load of a 3-D box at (x, y, z) of `map` into this CTA's shared
// memory at `dst` (16-byte aligned; x * 4 bytes a multiple of 16), completing
// on `bar`.  The box's bytes must have been announced on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// ----------------------------------------------------------------------------
// Kernel 1: persistent sampled
// ----------------------------------------------------------------------------

// One CTA owns a row for all three phases (section 5.5, "Persistent sampled"):
// Phase 1, the complete-row pass with its certification (band rescue, exact
// coarse recovery), and Phase 3.  Rows after the first wave are claimed from a
// device counter in completion order.
//
// The work of a row that is not a pass over the row is split between two warp
// groups that run at the same time: warps [0, kRefineWarps) refine and commit
// the row just classified, while the other warps claim the next row and run
// its Phase 1 (view histogram, boundaries and cutoffs, or the guess source)
// into a second slot and histogram.  The next row's complete-row pass then
// starts as soon as both groups are done.

// The persistent CTA's TMA view buffer: kViewBoxes boxes of 4 KB, their
// mbarrier and the barrier's phase word (bit 0: parity of the next phase;
// bit 1: a copy timed out, the buffer is not used again).
struct ViewDma {
  uint32_t* buf;
  uint32_t bar;
  uint32_t* phase;
};

// Phase 1's view (eq. 13) by group G through the TMA engine.  Box q of
// {4, box, 1} scores at (a & ~3, q * box, r) lands at buf + 1024 q, so view
// entry t is buf[1024 (t / box) + 4 (t % box) + (a & 3)].  Entries past the
// boxes (views longer than kViewBoxes boxes, or in the last partial line of a
// row whose capacity N is not a multiple of s) are loaded directly, as are all
// of them once a copy has timed out.  Entered with a cleared histogram; leaves
// it dirty.
// View entries of row r (length L, phase a) that the TMA boxes cover, and the
// number of boxes.
__device__ __forceinline__ int view_boxes(const Params& p, int L, int a, int& covered) {
  const int nv = view_size(L, a, p.s);
  const int box = p.view_box;
  covered = min(min(nv, p.N / p.s), (int)kViewBoxes * box);
  return (covered + box - 1) / box;
}

// Issues the view boxes of row r (one thread); false when nothing was issued.
__device__ __forceinline__ bool view_tma_issue(const Params& p, int r, int L, int a,
                                               const ViewDma& vd) {
  int covered;
  const int nq = view_boxes(p, L, a, covered);
  if ((*vd.phase & 2u) != 0u || nq <= 0) return false;
  // earlier generic reads of the buffer are ordered before the copies
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(vd.bar, (uint32_t)nq * (uint32_t)p.view_box * 16u);
  for (int q = 0; q < nq; ++q)
    tma_load_3d(smem_addr(vd.buf) + (uint32_t)q * 4096u, &p.view_map, a & ~3, q * p.view_box, r,
                vd.bar);
  return true;
}

template <class G>
__device__ void sample_view_tma(const Params& p, int r, const float* row, int L, int a,
                                uint32_t* hist, GroupScratch& sc, Slot& sl, const ViewDma& vd) {
  const int nv = view_size(L, a, p.s);
  const int tid = G::rank();
  const int box = p.view_box;
  int covered;
  (void)view_boxes(p, L, a, covered);
  if (tid == 0) {
    int ok = 0;
    if (view_tma_issue(p, r, L, a, vd)) {
      const uint32_t ph = *vd.phase & 1u;
      if (mbar_wait_parity_bounded(vd.bar, ph)) {
        *vd.phase = ph ^ 1u;
        ok = 1;
      } else {
        *vd.phase = 2u;  // copies may still land: the buffer is retired
        flag_status(p.counters, 4);
      }
    }
    sc.bcast = ok;
  }
  G::sync();
  const int lim = sc.bcast != 0 ? covered : 0;
  for (int t = tid; t < nv; t += G::kThreads) {
    const uint32_t u =
        t < lim ? vd.buf[1024 * (t / box) + 4 * (t % box) + (a & 3)]
                : __ldg(reinterpret_cast<const unsigned int*>(row) + a + (int64_t)t * p.s);
    smem_add(&hist[coarse_bin(u)], 1u);
  }
  G::sync();
  view_cutoffs<G>(p, hist, sc, sl);
}

// What Phase 1 left for a claimed row (Slot::route of the next-row slot).
constexpr int kNextNone = -1;    // the queue is exhausted
constexpr int kNextPad = 0;      // L <= K: padded output, no selection
constexpr int kNextSampled = 1;  // view cutoffs T0 (and T1) in the slot
constexpr int kNextDirect = 2;   // view too small: exact coarse recovery
constexpr int kNextGuess = 3;    // guess-source cutoff T0 in the slot
constexpr int kNextDeferred = 4; // handed to the heavy-row kernel (record in Params::defer)
// Slot::route of a row handed to the heavy-row epilogue after its Phase 2 count.
constexpr int kRouteDeferred = -1;

// A sampled row whose view predicts C(tau0) ~ s * (view entries in bins <=
// tau0) above four on-chip frontier capacities: a tie group, a constant row
// or a block of subnormals admitted whole.  Such a frontier costs as much to
// write and re-read as the row, and refining it in global memory takes more
// rounds than the passes over the row the heavy-row machinery makes.
__device__ __forceinline__ bool heavy_view(const Params& p, uint32_t vcnt) {
  return p.defer != nullptr && (uint64_t)vcnt * (uint64_t)p.s > 4ull * (uint64_t)p.cap;
}

// Hands row nr to the heavy-row epilogue of this CTA (one thread): its record
// {row, L, T0, T1, tau0, tau1} and its place in the CTA's list.
__device__ __forceinline__ void defer_row(const Params& p, uint32_t* own, int nr, int L, uint32_t T0,
                                          uint32_t T1, int tau0, int tau1) {
  const int i = atomicAdd(p.counters + kCtrDeferred, 1);
  int32_t* rec = p.defer + 8 * (int64_t)i;
  rec[0] = nr;
  rec[1] = L;
  rec[2] = (int32_t)T0;
  rec[3] = (int32_t)T1;
  rec[4] = tau0;
  rec[5] = tau1;
  own[1 + own[0]] = (uint32_t)i;
  own[0] = own[0] + 1u;
}

// Claims a row (or takes `assigned`) and runs its Phase 1 by group V into
// `nx`, with `vh` as the view histogram.  The caller publishes `nx` with a CTA
// barrier.
template <class V>
__device__ void prepare_row(const Params& p, int M, int assigned, Slot& nx, uint32_t* vh,
                            GroupScratch& sc, const ViewDma& vd) {
  if (V::rank() == 0) {
    const int nr = assigned >= 0 ? assigned : (int)gridDim.x + atomicAdd(p.counters + kCtrQueue, 1);
    sc.bcast = nr;
    sc.bcast2 = nr < M ? row_length(p, nr) : 0;
  }
  V::sync();
  const int nr = sc.bcast, L = sc.bcast2;
  int kind;
  if (nr >= M) {
    kind = kNextNone;
  } else if (L <= p.K) {
    kind = kNextPad;
  } else {
    const float* row = p.logits + (int64_t)nr * p.pitch;
    if (V::rank() == 0) {
      // the head of the row: in flight from HBM before its complete-row pass
      // (16-byte aligned range inside the row)
      const uintptr_t b = (reinterpret_cast<uintptr_t>(row) + 15u) & ~(uintptr_t)15u;
      const uintptr_t e = (reinterpret_cast<uintptr_t>(row) + (uintptr_t)L * 4u) & ~(uintptr_t)15u;
      if (e > b) {
        const uintptr_t len = e - b < kL2Next ? e - b : kL2Next;
        prefetch_l2(reinterpret_cast<const void*>(b), (uint32_t)len);
      }
    }
    if (p.prev != nullptr && guess_bin<V>(p, row, L, nr, sc, nx)) {
      kind = kNextGuess;
    } else {
      const int a = view_phase(nr, p.s, p.s_bits);
      if (view_size(L, a, p.s) >= (p.dual ? p.q1 : p.q0)) {
        clear_hist<V>(vh, 2048);
        V::sync();
        if (p.view_tma)
          sample_view_tma<V>(p, nr, row, L, a, vh, sc, nx, vd);
        else
          sample_view<V>(p, row, L, a, vh, sc, nx);
        kind = kNextSampled;
        // this CTA's list of deferred rows (persistent layout)
        uint32_t* own = reinterpret_cast<uint32_t*>(
            smem_base() + smem_layout(EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, kPersistentCap).own);
        if (heavy_view(p, nx.vcnt0) && own[0] < kMaxOwnDeferred) {
          // the rest of this row's method runs in the CTA's epilogue
          // (finish_deferred), after its other rows
          V::sync();  // every thread has read own[0]
          if (V::rank() == 0) defer_row(p, own, nr, L, nx.T0, nx.T1, nx.tau0, nx.tau1);
          kind = kNextDeferred;
        }
      } else {
        kind = kNextDirect;
      }
    }
  }
  if (V::rank() == 0) {
    nx.row = nr;
    nx.L = L;
    nx.route = kind;
  }
}

// One row whose Phase 1 sits in `nx`; on return `nx` holds the next row's.
// Entered and left at a CTA barrier.
__device__ void persistent_row(const Params& p, int M, Slot& sl, Slot& nx, const Frontier& F,
                               uint32_t* hist, uint32_t* vhist, GroupScratch* sc2,
                               uint32_t* queues, const ViewDma& vd) {
  using G = CtaGroup<kPersistentThreads>;
  using R = SubGroup<kRefineWarps * 32, 0, 1>;
  using V = SubGroup<kPersistentThreads - kRefineWarps * 32, kRefineWarps, 2>;
  GroupScratch& sc = sc2[0];
  const int K = p.K;
  const int r = nx.row, L = nx.L, kind = nx.route;
  const uint32_t T0 = nx.T0, T1 = nx.T1;
  const int tau0 = nx.tau0, tau1 = nx.tau1;
  const float* row = p.logits + (int64_t)r * p.pitch;
  int32_t* out_row = p.out + (int64_t)r * K;
  const bool idle = kind == kNextPad || kind == kNextDeferred;  // no selection work here
  if (!idle) clear_hist<G>(hist, 2048);
  if (threadIdx.x == 0) {
    sl.row = r;
    sl.L = L;
    sl.n_front = 0u;
    sl.n_out = 0u;
    sl.n_drop = 0u;
    sl.T0 = T0;
    sl.T1 = T1;
    sl.tau0 = kind == kNextSampled || kind == kNextGuess ? tau0 : -1;
    sl.tau1 = kind == kNextSampled ? tau1 : -1;
    sl.c0 = -1;
    sl.c1 = -1;
    sl.tstar = -1;
    sl.e0 = 0;
    sl.vcnt1 = kind == kNextSampled ? nx.vcnt1 : 0u;
  }
  __syncthreads();  // every thread has read nx; the next row's group may overwrite it
  if (kind == kNextPad) {
    write_pad_row<G>(out_row, L, K);
    if (threadIdx.x == 0) write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
  } else if (kind == kNextDeferred) {
    // written by the heavy-row kernel
  } else {
    FrontierSink front_sink{{}, F, hist};
    DropSink drop;
    int route;
    if (kind == kNextGuess) {
      scan_two_class<G>(row, 0, L, T0, T0, false, &sl.n_drop, &sl.n_front, queues, drop,
                        front_sink);
      G::sync();
      const uint32_t c0 = sl.n_front;
      route = c0 >= (uint32_t)K ? EXACT_TOPK_ROUTE_GUESS : EXACT_TOPK_ROUTE_GUESS_EXACT;
      if (threadIdx.x == 0) sl.c0 = (int)c0;
    } else if (kind == kNextSampled) {
      // Phase 2: admit d <= T0, persist candidates, build h0 (eqs. 16-17).
      scan_two_class<G>(row, 0, L, T0, T0, false, &sl.n_drop, &sl.n_front, queues, drop,
                        front_sink);
      G::sync();
      const uint32_t c0 = sl.n_front;
      if (c0 >= (uint32_t)K) {
        route = EXACT_TOPK_ROUTE_PRIMARY;
      } else if (p.dual) {
        uint32_t* own = reinterpret_cast<uint32_t*>(
            smem_base() + smem_layout(EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, kPersistentCap).own);
        if (heavy_view(p, sl.vcnt1) && own[0] < kMaxOwnDeferred) {
          // the view puts the band far beyond on-chip capacity: the rest of
          // the row's method runs in the CTA's epilogue (which counts C(tau0)
          // again)
          G::sync();  // every thread has read own[0]
          if (threadIdx.x == 0) defer_row(p, own, r, L, T0, T1, tau0, tau1);
          route = kRouteDeferred;
        } else {
          // Band rescue (eqs. 18-19): a second pass appends only T0 < d <= T1.
          if (T1 > T0)
            scan_two_class<G>(row, 0, L, T0, T1, true, &sl.n_drop, &sl.n_front, queues, drop,
                              front_sink);
          G::sync();
          const uint32_t c1 = sl.n_front;
          route = c1 >= (uint32_t)K ? EXACT_TOPK_ROUTE_BAND : EXACT_TOPK_ROUTE_EXACT_AFTER_BAND;
          if (threadIdx.x == 0) sl.c1 = (int)c1;
        }
      } else {
        route = EXACT_TOPK_ROUTE_EXACT_NO_BAND;
      }
      if (threadIdx.x == 0) sl.c0 = (int)c0;
    } else {
      route = EXACT_TOPK_ROUTE_DIRECT_EXACT;
    }
    const bool exact =
        route == EXACT_TOPK_ROUTE_EXACT_AFTER_BAND || route == EXACT_TOPK_ROUTE_EXACT_NO_BAND ||
        route == EXACT_TOPK_ROUTE_GUESS_EXACT || route == EXACT_TOPK_ROUTE_DIRECT_EXACT;
    if (threadIdx.x == 0) {
      sl.route = route;
      sl.q0n = (int)sl.n_front;  // eq. 21: E0 = {}, Q0 = A(tau), k0 = K
    }
    G::sync();
    if (exact) {
      // the last cutoff Phase 2 tried (T1 when the band widened T0)
      const bool band = tau1 > tau0;
      if (kind != kNextSampled ||
          !bounded_recovery<G>(p, row, L, F, hist, vhist, sc, sl, queues, band ? T1 : T0,
                               band ? tau1 : tau0))
        exact_recovery<G>(p, row, L, F, hist, sc, sl, out_row, queues);
    }
  }
  // Phase 3 of this row and Phase 1 of the next: side by side when the
  // frontier is in shared memory; one after the other, each by the whole CTA,
  // when it spilled (refinement then streams the global slice and wants every
  // warp) or when there is nothing to refine.
  const bool busy = !idle && sl.route != kRouteDeferred;  // a row deferred at its band: none
  const bool split = busy && sl.n_front <= F.cap;
  if (split) {
    if ((int)(threadIdx.x >> 5) < kRefineWarps) {
      refine<R>(F, sl.n_front, (uint32_t)K - sl.n_out, hist, sc, sl, out_row, K, queues,
                (uint32_t)(R::kWarps * kQueueWords));
      finish_row<R>(p, sl, out_row);
      if (threadIdx.x == 0) write_slot_trace(p, sl);
    } else {
      prepare_row<V>(p, M, -1, nx, vhist, sc2[1], vd);
    }
  } else {
    if (busy) {
      refine<G>(F, sl.n_front, (uint32_t)K - sl.n_out, hist, sc, sl, out_row, K, queues,
                (uint32_t)(G::kWarps * kQueueWords));
      finish_row<G>(p, sl, out_row);
      if (threadIdx.x == 0) write_slot_trace(p, sl);
    }
    prepare_row<G>(p, M, -1, nx, vhist, sc2[1], vd);
  }
  __syncthreads();
}

// Finishes the rows this CTA deferred (defined with the heavy-row machinery).
__device__ __noinline__ void finish_deferred(const Params& p);

__global__ void __launch_bounds__(kPersistentThreads, 1024 / kPersistentThreads)
    persistent_sampled_kernel(const __grid_constant__ Params p) {
  unsigned char* sm = smem_base();
  constexpr SmemLayout lay = smem_layout(EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, kPersistentCap);
  Slot* slots = reinterpret_cast<Slot*>(sm + lay.slots);  // [0] this row, [1] the next
  GroupScratch* sc2 = reinterpret_cast<GroupScratch*>(sm + lay.scratch);
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + lay.hist);
  uint32_t* vhist = hist + kCoarseBins;
  uint32_t* queues = reinterpret_cast<uint32_t*>(sm + lay.queues);
  const Frontier F = make_frontier(p, reinterpret_cast<uint2*>(sm + lay.frontier), blockIdx.x);
  const ViewDma vd{reinterpret_cast<uint32_t*>(sm + lay.vbuf), smem_addr(sm + lay.vbar),
                   reinterpret_cast<uint32_t*>(sm + lay.vbar + 8)};
  const int M = live_rows(p);
  if ((int)blockIdx.x < M) {  // CTA-uniform
    if (threadIdx.x == 0) {
      mbar_init(vd.bar, 1u);
      // the boxes' shared destination must be 128-byte aligned: otherwise the
      // buffer is retired from the start and the view is gathered directly
      *vd.phase = (smem_addr(vd.buf) & 127u) == 0u ? 0u : 2u;
      *reinterpret_cast<uint32_t*>(sm + lay.own) = 0u;
    }
    __syncthreads();
    prepare_row<CtaGroup<kPersistentThreads>>(p, M, (int)blockIdx.x, slots[1], vhist, sc2[1], vd);
    __syncthreads();
    while (slots[1].route != kNextNone)
      persistent_row(p, M, slots[0], slots[1], F, hist, vhist, sc2, queues, vd);
    if (*reinterpret_cast<const uint32_t*>(smem_base() + lay.own) != 0u) finish_deferred(p);
  }
  exit_protocol(p.counters);
}

// ----------------------------------------------------------------------------
// Kernel 2: row-local exact
// ----------------------------------------------------------------------------

__global__ void __launch_bounds__(kRowLocalThreads, 1) row_local_exact_kernel(Params p) {
  using G = CtaGroup<kRowLocalThreads>;
  unsigned char* sm = smem_base();
  constexpr SmemLayout lay = smem_layout(EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT, kRowLocalCap);
  Slot& sl = *reinterpret_cast<Slot*>(sm + lay.slots);
  GroupScratch& sc = *reinterpret_cast<GroupScratch*>(sm + lay.scratch);
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + lay.hist);
  uint32_t* queues = reinterpret_cast<uint32_t*>(sm + lay.queues);
  const Frontier F = make_frontier(p, reinterpret_cast<uint2*>(sm + lay.frontier), blockIdx.x);
  const int M = live_rows(p);
  int r = blockIdx.x;
  while (r < M) {
    const int K = p.K;
    const float* row = p.logits + (int64_t)r * p.pitch;
    const int L = row_length(p, r);
    int32_t* out_row = p.out + (int64_t)r * K;
    if (L <= K) {
      write_pad_row<G>(out_row, L, K);
      if (threadIdx.x == 0) write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    } else {
      if (L <= kRowLocalResident)
        exact_recovery_resident<G, kRowLocalResident / kRowLocalThreads>(p, row, L, F, hist, sc,
                                                                          sl, out_row);
      else
        exact_recovery<G>(p, row, L, F, hist, sc, sl, out_row, queues);
      refine<G>(F, sl.n_front, (uint32_t)(K - sl.e0), hist, sc, sl, out_row, K, queues,
              (uint32_t)(G::kWarps * kQueueWords));
      finish_row<G>(p, sl, out_row);
      if (threadIdx.x == 0)
        write_trace(p, r, EXACT_TOPK_ROUTE_DIRECT_EXACT, -1, -1, -1, -1, sl.tstar, sl.e0, sl.q0n);
    }
    __syncthreads();
    if (threadIdx.x == 0) sc.bcast = (int)gridDim.x + atomicAdd(p.counters + kCtrQueue, 1);
    __syncthreads();
    r = sc.bcast;
    __syncthreads();
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
struct SegmentFrontSink : NoCount {
  uint2* rb;
  int lo;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    rb[lo + (int)p] = make_uint2((uint32_t)i, d);
  }
};
struct SegmentBackSink : NoCount {
  uint2* rb;
  int hi;
  __device__ __forceinline__ void operator()(uint32_t p, int32_t i, uint32_t d) const {
    rb[hi - 1 - (int)p] = make_uint2((uint32_t)i, d);
  }
};

__global__ void __launch_bounds__(kKvSplitThreads, 2) kv_split_kernel(Params p) {
  using G = CtaGroup<kKvSplitThreads>;
  unsigned char* sm = smem_base();
  constexpr SmemLayout lay = smem_layout(EXACT_TOPK_FAMILY_KV_SPLIT, kKvSplitCap);
  Slot& sl = *reinterpret_cast<Slot*>(sm + lay.slots);
  GroupScratch& sc = *reinterpret_cast<GroupScratch*>(sm + lay.scratch);
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + lay.hist);
  uint32_t* run_pre = reinterpret_cast<uint32_t*>(sm + lay.runs);
  uint32_t* run_c0 = run_pre + kMaxSplits + 1;
  uint32_t* run_cb = run_c0 + kMaxSplits;
  uint32_t* queues = reinterpret_cast<uint32_t*>(sm + lay.queues);
  const int r = blockIdx.y;
  const int seg = blockIdx.x;
  const int P = p.P;
  const int K = p.K;
  const int tid = threadIdx.x;
  if (r >= live_rows(p)) return;
  const float* row = p.logits + (int64_t)r * p.pitch;
  const int L = row_length(p, r);
  int32_t* out_row = p.out + (int64_t)r * K;
  // Row buffer: segment-owned candidate ranges, later the finisher's spill.
  uint2* rb = p.ws + (int64_t)r * p.N;
  const Frontier F = make_frontier(p, reinterpret_cast<uint2*>(sm + lay.frontier), r);

  if (L <= K) {
    if (seg == 0) {
      write_pad_row<G>(out_row, L, K);
      if (tid == 0) write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    }
    return;
  }
  clear_hist<G>(hist, 2048);
  if (tid == 0) {
    sl.seg_c0 = 0u;
    sl.seg_cb = 0u;
    sl.n_front = 0u;
    sl.n_out = 0u;
    sl.tau0 = -1;
    sl.tau1 = -1;
    sl.e0 = 0;
    sl.tstar = -1;
  }
  G::sync();

  // Every segment reconstructs the same row-local proposal from r alone.
  bool guess = false;
  uint32_t T0 = 0u, T1 = 0u;
  bool use_band = false;
  if (p.prev != nullptr && guess_bin<G>(p, row, L, r, sc, sl)) {
    guess = true;
    T0 = sl.T0;
  } else {
    const int a = view_phase(r, p.s, p.s_bits);
    const int qmax = p.dual ? p.q1 : p.q0;
    if (view_size(L, a, p.s) < qmax) {
      // View unusable: the row takes the direct-exact route on one CTA.
      if (seg == 0) {
        exact_recovery<G>(p, row, L, F, hist, sc, sl, out_row, queues);
        refine<G>(F, sl.n_front, (uint32_t)(K - sl.e0), hist, sc, sl, out_row, K, queues,
              (uint32_t)(G::kWarps * kQueueWords));
        finish_row<G>(p, sl, out_row);
        if (tid == 0)
          write_trace(p, r, EXACT_TOPK_ROUTE_DIRECT_EXACT, -1, -1, -1, -1, sl.tstar, sl.e0,
                      sl.q0n);
      }
      return;
    }
    sample_view<G>(p, row, L, a, hist, sc, sl);
    T0 = sl.T0;
    T1 = sl.T1;
    use_band = p.dual && T1 > T0;
  }
  const int tau0 = sl.tau0, tau1 = guess ? -1 : sl.tau1;

  // Phase 2 over this segment, with the band (T0 < d <= T1) collected in the
  // same traversal: an underfilled primary needs no second pass.
  int lo, hi;
  segment_bounds(L, P, seg, lo, hi);
  {
    SegmentFrontSink primary{{}, rb, lo};
    SegmentBackSink band{{}, rb, hi};
    scan_two_class<G>(row, lo, hi, T0, use_band ? T1 : T0, true, &sl.seg_c0, &sl.seg_cb, queues,
                      primary, band);
  }
  __threadfence();  // every writer publishes its candidates before the arrival
  G::sync();
  if (tid == 0) {
    int32_t* counts = p.seg_counts + ((int64_t)r * P + seg) * 2;
    counts[0] = (int32_t)sl.seg_c0;
    counts[1] = (int32_t)sl.seg_cb;
    __threadfence();
    const int prev = atomicAdd(p.counters + kCtrArriveBase + r, 1);
    sl.is_last = prev == P - 1;
  }
  G::sync();
  if (!sl.is_last) return;

  // ---- finisher: merge (eq. 27), certify, refine or recover ----
  __threadfence();
  if (tid == 0) atomicExch(p.counters + kCtrArriveBase + r, 0);
  for (int q = tid; q < P; q += kKvSplitThreads) {
    const int32_t* cq = p.seg_counts + ((int64_t)r * P + q) * 2;
    run_c0[q] = (uint32_t)__ldcg(cq);
    run_cb[q] = (uint32_t)__ldcg(cq + 1);
  }
  G::sync();
  if (tid < 32) {
    // Totals of both counts, each lane summing up to 4 consecutive segments.
    uint32_t s0 = 0u, sb = 0u;
    for (int q = tid * 4; q < tid * 4 + 4 && q < P; ++q) {
      s0 += run_c0[q];
      sb += run_cb[q];
    }
    s0 = __reduce_add_sync(kFull, s0);
    sb = __reduce_add_sync(kFull, sb);
    if (tid == 0) {
      sl.c0 = (int)s0;
      sl.c1 = (int)sb;
    }
  }
  G::sync();
  const uint32_t c0 = (uint32_t)sl.c0, cb = (uint32_t)sl.c1;
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
        run_pre[q] = acc;
        acc += run_c0[q] + (with_band ? run_cb[q] : 0u);
      }
      run_pre[P] = acc;
    }
    clear_hist<G>(hist, 2048);
    G::sync();
    // Gather the runs into the frontier in order.  Logical position f maps to
    // shared memory below cap and to rb[f] above; every source position is >=
    // its logical position, so gathering in chunks (read all, then write)
    // never overwrites an unread entry.
    const uint32_t total = run_pre[P];
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
            if (run_pre[mid] <= g)
              lo_q = mid;
            else
              hi_q = mid - 1;
          }
          const int q = lo_q;
          int slo, shi;
          segment_bounds(L, P, q, slo, shi);
          const uint32_t off = g - run_pre[q];
          const uint32_t n0 = run_c0[q];
          // band entries occupy [shi - nb, shi); read them in ascending order
          // so that every source position is >= its logical position
          const int src = off < n0 ? slo + (int)off : shi - (int)run_cb[q] + (int)(off - n0);
          const uint2 e = __ldcg(rb + src);
          idx[k] = (int32_t)e.x;
          key[k] = e.y;
        }
      }
      G::sync();
#pragma unroll
      for (int k = 0; k < R; ++k) {
        if (idx[k] == -2) continue;
        F.put(c + k * kKvSplitThreads + tid, idx[k], key[k]);
        atomicAdd(&hist[key[k] >> 21], 1u);
      }
      G::sync();
    }
    q0n = (int)total;
    refine<G>(F, total, (uint32_t)K, hist, sc, sl, out_row, K, queues,
              (uint32_t)(G::kWarps * kQueueWords));
  } else {
    exact_recovery<G>(p, row, L, F, hist, sc, sl, out_row, queues);
    tstar = sl.tstar;
    e0 = sl.e0;
    q0n = sl.q0n;
    refine<G>(F, sl.n_front, (uint32_t)(K - e0), hist, sc, sl, out_row, K, queues,
              (uint32_t)(G::kWarps * kQueueWords));
  }
  finish_row<G>(p, sl, out_row);
  if (tid == 0) write_trace(p, r, route, tau0, tau1, (int)c0, c1, tstar, e0, q0n);
}

// ----------------------------------------------------------------------------
// Kernel 4: cluster-resident split (section 4.5 eqs. 26-27, merge made on chip)
// ----------------------------------------------------------------------------
//
// The P CTAs of one thread-block cluster own one row.  Each CTA copies its
// segment (at most kClusterStage scores) into shared memory with one TMA bulk
// copy, issued right after the loads of the replicated Phase-1 view so that
// the copy overlaps the view.  Phase 2 is one pass over the resident segment
// that counts both classes and writes each admitted key with its position to
// the warp's region (ranks from ballots, no atomics).  After one cluster
// barrier every CTA reads the counts of eq. 27, takes the same route, gathers
// the frontier keys of all CTAs through distributed shared memory and selects
// the K-th smallest frontier key locally; each CTA then commits its own
// entries below that key and its share of the ties, with output ranges
// reserved by one atomic pair on the leader CTA.  Frontiers that do not fit
// the merged list (tie runs, constant rows) and exact coarse recovery run the
// 11+11+10 recurrence with cluster-summed histograms over the resident
// segments, so no route re-reads HBM.

// Per-CTA shared state of the cluster kernel (at offset 0 of dynamic smem).
struct ClusterState {
  uint64_t bar;        // mbarrier of the segment copy
  uint32_t cnt_a;      // |{d <= T0}| in this segment
  uint32_t cnt_b;      // |{T0 < d <= T1}| in this segment
  uint32_t n_out;      // leader: output slots handed out
  uint32_t n_keep;     // leader: tie slots handed out
  int32_t timed_out;   // the segment copy did not complete in time
  uint32_t kmin;       // smallest admitted key (d <= T1) in this segment
  int32_t pad_[4];
  uint32_t wcnt[16];   // admitted keys (d <= T1) found by each warp
  uint32_t pad2_[16];
};
static_assert(sizeof(ClusterState) % 16 == 0, "ClusterState keeps the layout 16-byte aligned");

// Admitted (key, position) pairs each warp of a cluster CTA can hold; the
// merged list of a row holds at most kMergeCap keys.  Larger frontiers (tie runs, constant
// rows) take the histogram path over the resident segments.
constexpr int kRegionCap = 128;
constexpr uint32_t kMergeCap = 3 * kCoarseBins;

struct ClusterLayout {
  uint32_t state, slot, scratch, h256, hist, keys, pos, sumx, stage, total;
};
__host__ __device__ constexpr ClusterLayout cluster_layout() {
  ClusterLayout l{};
  uint32_t o = 0;
  l.state = o;
  o = align16(o + (uint32_t)sizeof(ClusterState));
  l.slot = o;
  o = align16(o + (uint32_t)sizeof(Slot));
  l.scratch = o;
  o = align16(o + 2 * (uint32_t)sizeof(GroupScratch));
  l.h256 = o;  // private: region offsets and counts of the merged list
  o = align16(o + 256u * 4u);
  l.hist = o;  // private 2048-bin histogram of the selections
  o = align16(o + kCoarseBins * 4u);
  l.keys = o;  // published: per-warp regions of admitted keys (fallback: an exchange histogram)
  o = align16(o + (kClusterThreads / 32) * kRegionCap * 4u);
  l.pos = o;   // private: their segment positions
  o = align16(o + (kClusterThreads / 32) * kRegionCap * 2u);
  l.sumx = o;  // private merged frontier; or [summed histogram | published exchange histogram]
  o = align16(o + kMergeCap * 4u);
  o = (o + 127u) & ~127u;
  l.stage = o;  // the resident segment
  o += kClusterStage * 4u;
  l.total = o;
  return l;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Full cluster barrier with release/acquire ordering of shared memory.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
  return a;
}
// Peer loads are volatile (they stay in order with the cluster barriers, which
// clobber memory) but carry no memory clobber of their own, so independent
// loads can be in flight together.
__device__ __forceinline__ uint4 ld_peer4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t ld_peer(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t atom_add_peer(uint32_t a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_peer(uint32_t a, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
// Sums histogram `local` (nbins, a multiple of 4, at most 4 per thread) over
// the P CTAs of the cluster into `sum`.  Group barrier before return.
template <class G>
__device__ __forceinline__ void cluster_hist_sum(const uint32_t* local, uint32_t* sum, int nbins,
                                                 int P) {
  const int t = G::rank();
  if (4 * t < nbins) {
    const uint32_t la = smem_addr(local + 4 * t);
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
    for (int q = 0; q < P; ++q) {
      const uint4 v = ld_peer4(peer_addr(la, (uint32_t)q));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<uint4*>(sum + 4 * t) = acc;
  }
  G::sync();
}

// The frontier of the cluster kernel is a key interval: lo_open < d <= hi
// (lo_open absent on the sampled routes).  Keys at or below lo_open are the
// E0 of exact coarse recovery (committed outright).
struct KeyBand {
  uint32_t lo;  // exclusive lower key bound
  uint32_t hi;  // inclusive upper key bound
  bool has_lo;
  __device__ __forceinline__ bool in(uint32_t d) const { return d <= hi && (!has_lo || d > lo); }
  __device__ __forceinline__ bool below(uint32_t d) const { return has_lo && d <= lo; }
};

// Screen of four staged scores against an inclusive key bound T: false only
// when none of them can have key <= T.  For a non-negative cutoff score the
// key order on candidates is the signed order of the raw bits.
struct Screen {
  uint32_t T;
  int C;
  bool fast;
  __device__ __forceinline__ explicit Screen(uint32_t T_) : T(T_) {
    const uint32_t b = bits_from_desc(T_);
    fast = (b & 0x80000000u) == 0u;
    C = (int)b;
  }
  __device__ __forceinline__ bool any(const uint4& v) const {
    if (fast) return max(max((int)v.x, (int)v.y), max((int)v.z, (int)v.w)) >= C;
    return min(min(desc_key(v.x), desc_key(v.y)), min(desc_key(v.z), desc_key(v.w))) <= T;
  }
};


// Result of Phase 3: commit every frontier key below `commit_below`, then
// `ties` keys equal to `tie_key`.
struct Cut {
  uint64_t commit_below;
  uint32_t tie_key;
  uint32_t ties;
  bool bad;
};

// Phase 3 over the cluster for rows whose frontier does not fit a merged
// list (tie-heavy rows, exact coarse recovery).  Each round histograms an
// 11-bit digit taken over the candidate key interval [qlo, qhi) (initially
// the frontier's interval: (F.lo, F.hi], or [lo_hint, F.hi] without a lower
// bound), sums it over the cluster through DSMEM and narrows the interval to
// the boundary bucket; the threshold is the one eqs. 22-25 reach with fixed
// 11+11+10 digits.  A frontier inside one coarse bin (exact recovery) spans
// about 2^18 keys and resolves in two rounds.  `xa` and `xc` alternate as the
// published buffer; `sum` is private.
template <class G, class Vec>
__device__ Cut cluster_select(const Vec& seg_vec, int n, const KeyBand& F, uint32_t k,
                              uint32_t* xa, uint32_t* xc, uint32_t* sum, GroupScratch& sc, int P,
                              uint32_t lo_hint) {
  const int tid = G::rank();
  const int nv4 = (n + 3) >> 2;
  Cut cut{0, 0u, 0u, false};
  uint64_t qlo = F.has_lo ? (uint64_t)F.lo + 1u : (uint64_t)lo_hint;  // inclusive
  uint64_t qhi = (uint64_t)F.hi + 1u;                                  // exclusive
  uint32_t* nxt = xa;
  for (int round = 0; round < 4; ++round) {  // 32 bits in 11-bit digits: 3 rounds suffice
    if (qhi <= qlo) {
      cut.bad = true;
      return cut;
    }
    if (qhi - qlo == 1u) {
      // one key value left: the k remaining entries are ties (eq. 25)
      cut.commit_below = qlo;
      cut.tie_key = (uint32_t)qlo;
      cut.ties = k;
      return cut;
    }
    const int bits = 64 - __clzll((long long)(qhi - qlo - 1u));
    const int width = bits < 11 ? bits : 11;
    const int shift = bits - width;
    const int nbins = (1 << width) < 128 ? 128 : (1 << width);
    clear_hist<G>(nxt, nbins);
    G::sync();
    {
      const Screen scr((uint32_t)(qhi - 1u));
      RunHist rh;
      for (int t = tid; t < nv4; t += G::kThreads) {
        const uint4 v = seg_vec(t);
        if (!scr.any(v)) continue;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t d = desc_key(u[e]);
          if (4 * t + e < n && (uint64_t)d >= qlo && (uint64_t)d < qhi)
            rh.add(nxt, (uint32_t)(((uint64_t)d - qlo) >> shift));
        }
      }
      rh.flush(nxt);
    }
    G::sync();
    cluster_sync_all();
    cluster_hist_sum<G>(nxt, sum, nbins, P);
    nxt = nxt == xa ? xc : xa;
    find_boundaries<G>(sum, sc, nbins, 1, k, 0u);
    const int b = sc.res_bin[0];
    const uint32_t below = sc.res_below[0], cnt = sc.res_cnt[0];
    if (b < 0) {
      cut.bad = true;
      return cut;
    }
    qlo += (uint64_t)b << shift;
    const uint64_t top = qlo + ((uint64_t)1 << shift);
    qhi = top < qhi ? top : qhi;
    if (below + cnt == k) {
      // the boundary bucket closes the quota: every key below its end
      cut.commit_below = qhi;
      return cut;
    }
    k -= below;
  }
  cut.bad = true;
  return cut;
}

// Commit of a cluster CTA: every accepted key goes to
// [0, K - ties), the first `ties` keys equal to the tie key to [K - ties, K)
// over the cluster.  A block scan of the per-thread counts gives every thread
// its offsets and each CTA reserves its ranges with one atomic pair on the
// leader's counters, so placing the entries needs no atomics.  `visit(pass,
// fn)` calls fn(key, index) for this thread's candidate entries, in the same
// order on both passes.
template <class G, class Visit>
__device__ void cluster_commit(const Visit& visit, uint64_t commit_below, uint32_t tie_key,
                               uint32_t ties, bool bad, uint32_t n_out_addr, uint32_t n_keep_addr,
                               GroupScratch& sc, int32_t* out_row, int K) {
  const int tid = G::rank();
  uint32_t nc = 0u, nt = 0u;
  if (!bad) {
    visit([&](uint32_t d, bool e0, int32_t) {
      if (e0 || (uint64_t)d < commit_below)
        ++nc;
      else if (ties > 0u && d == tie_key)
        ++nt;
    });
  }
  uint32_t tot;
  const uint32_t ex = block_exclusive_scan<G>(nc | (nt << 16), sc, tot);
  if (tid == 0) {
    const uint32_t NC = tot & 0xFFFFu, NT = tot >> 16;
    const uint32_t bc = NC ? atom_add_peer(n_out_addr, NC) : 0u;
    const uint32_t bt = NT ? atom_add_peer(n_keep_addr, NT) : 0u;
    sc.res_below[0] = bc;                       // first commit slot
    sc.res_below[1] = (uint32_t)K - ties + bt;  // first tie slot
    sc.res_cnt[1] = bt >= ties ? 0u : min(NT, ties - bt);  // ties this CTA fills
  }
  G::sync();
  if (!bad && (nc | nt) != 0u) {
    uint32_t oc = sc.res_below[0] + (ex & 0xFFFFu);
    uint32_t ot = ex >> 16;
    const uint32_t tbase = sc.res_below[1], take = sc.res_cnt[1];
    visit([&](uint32_t d, bool e0, int32_t idx) {
      if (e0 || (uint64_t)d < commit_below) {
        if (oc < (uint32_t)K) out_row[oc] = idx;
        ++oc;
      } else if (ties > 0u && d == tie_key) {
        if (ot < take && tbase + ot < (uint32_t)K) out_row[tbase + ot] = idx;
        ++ot;
      }
    });
  }
}

__global__ void __launch_bounds__(kClusterThreads, 2) cluster_split_kernel(Params p) {
  using G = CtaGroup<kClusterThreads>;
  static_assert(kClusterThreads / 32 == 16, "the merged-list table assumes 16 warps per CTA");
  static_assert(16 * kClusterMaxSplits <= 256 && (16 * kClusterMaxSplits) % 32 == 0,
                "sub-list table of 256 entries");
  unsigned char* sm = smem_base();
  constexpr ClusterLayout lay = cluster_layout();
  ClusterState& cs = *reinterpret_cast<ClusterState*>(sm + lay.state);
  Slot& sl = *reinterpret_cast<Slot*>(sm + lay.slot);
  GroupScratch& sc = *reinterpret_cast<GroupScratch*>(sm + lay.scratch);
  uint32_t* h256 = reinterpret_cast<uint32_t*>(sm + lay.h256);  // merged-list offsets
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + lay.hist);  // private
  uint32_t* keys = reinterpret_cast<uint32_t*>(sm + lay.keys);  // [kWarps][kRegionCap]
  uint16_t* pos = reinterpret_cast<uint16_t*>(sm + lay.pos);    // [kWarps][kRegionCap]
  uint32_t* sumx = reinterpret_cast<uint32_t*>(sm + lay.sumx);  // [kMergeCap]
  uint32_t* stage = reinterpret_cast<uint32_t*>(sm + lay.stage);
  uint32_t* sum = sumx;                  // summed histogram (private)
  uint32_t* xC = sumx + kCoarseBins;     // published: view samples or a histogram
  uint32_t* xA = keys;                   // published histogram on the fallback paths
  const int r = blockIdx.y;
  const uint32_t q = cluster_ctarank();
  const int P = p.P;
  const int K = p.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  // Every CTA of a cluster shares r, so these exits are cluster-uniform.
  if (r >= live_rows(p)) return;
  const float* row = p.logits + (int64_t)r * p.pitch;
  const int L = row_length(p, r);
  int32_t* out_row = p.out + (int64_t)r * K;
  if (L <= K) {
    if (q == 0) {
      write_pad_row<G>(out_row, L, K);
      if (tid == 0) write_trace(p, r, EXACT_TOPK_ROUTE_PAD, -1, -1, -1, -1, -1, -1, -1);
    }
    return;
  }
  int lo, hi;
  segment_bounds(L, P, (int)q, lo, hi);
  int n = hi - lo;  // <= kClusterSegment by the plan (checked on the host)
  if (n > kClusterSegment) {
    n = kClusterSegment;  // never taken for a valid plan; the row's result is flagged
    if (threadIdx.x == 0) flag_status(p.counters, 1);
  }
  const float* src = row + lo;
  const bool bulk = (reinterpret_cast<uintptr_t>(src) & 15u) == 0u;
  // The first `held` scores of the segment are held in shared memory; the
  // rest (segments longer than kClusterStage) are read from global memory,
  // prefetched into L2 while Phase 1 runs.
  const int held = n < kClusterStage ? n : kClusterStage;
  const int nb = bulk ? (held & ~3) : 0;  // scores moved by the bulk copy
  const uint32_t bar = smem_addr(&cs.bar);

  // Phase-1 view (eq. 13), replicated in every CTA of the cluster as in the
  // KV-split of section 4.5: its loads are issued ahead of the segment copy so
  // that they do not queue behind it.
  const int a = view_phase(r, p.s, p.s_bits);
  const int vsize = view_size(L, a, p.s);
  const bool sampled = p.prev == nullptr && vsize >= (p.dual ? p.q1 : p.q0);
  // Small clusters replicate the view in every CTA; clusters of more than
  // four CTAs split it: each CTA loads the view entries inside its own
  // segment and adds them into the leader's histogram (the union over the
  // segments is the row's view, eq. 13).
  const bool split_view = sampled && P > 4;
  int vt0 = 0, vt1 = vsize;  // view entries t in [vt0, vt1) handled here
  if (split_view) {
    vt0 = lo <= a ? 0 : (lo - a + p.s - 1) / p.s;
    vt1 = hi <= a ? 0 : min(vsize, (hi - a + p.s - 1) / p.s);
  }
  constexpr int kViewAhead = 8;  // view loads per thread issued before the copy
  uint32_t vu[kViewAhead];
#pragma unroll
  for (int k = 0; k < kViewAhead; ++k) {
    const int t = vt0 + k * G::kThreads + tid;
    vu[k] = (sampled && t < vt1)
                ? __ldg(reinterpret_cast<const unsigned int*>(row) + a + (int64_t)t * p.s)
                : 0u;
  }

  // ---- segment copy (TMA bulk) ----
  // Issued at once on the guess and direct routes; on the sampled route
  // (ETK_TMA_AFTER_VIEW) only once the view's loads have returned, so that
  // those loads do not queue behind the cluster's copies.
#ifndef ETK_TMA_AFTER_VIEW
#define ETK_TMA_AFTER_VIEW 0
#endif
  const bool copy_late = ETK_TMA_AFTER_VIEW && sampled;
  if (tid == 0) {
    mbar_init(bar, 1u);
    if (nb > 0 && !copy_late) bulk_copy_g2s(smem_addr(stage), src, (uint32_t)nb * 4u, bar);
    const uint32_t tail_bytes = (uint32_t)(n - held) * 4u & ~15u;
    if (bulk && tail_bytes > 0u) prefetch_l2(src + held, tail_bytes);
    cs.cnt_a = 0u;
    cs.cnt_b = 0u;
    cs.n_out = 0u;
    cs.n_keep = 0u;
    cs.timed_out = 0;
    cs.kmin = 0xFFFFFFFFu;
    sl.tau0 = -1;
    sl.tau1 = -1;
  }
  for (int t = nb + tid; t < held; t += G::kThreads) stage[t] = ld_stream1(src + t);

  // ---- Phase 1 ----
  // Every CTA histograms the whole row's view (replicated, as the KV-split of
  // section 4.5 does) and derives tau0 / tau1 and their cutoffs; the optional
  // guess source gathers its K scores instead.
  bool guess = false, direct = false;
  if (p.prev != nullptr && guess_bin<G>(p, row, L, r, sc, sl)) {
    guess = true;
  } else {
    direct = vsize < (p.dual ? p.q1 : p.q0);
  }
  if (!guess && !direct && split_view) {
    // Every CTA clears its exchange histogram before any CTA adds into the
    // leader's (first cluster barrier); the second orders the adds before
    // the reads.
    clear_hist<G>(xC, kCoarseBins);
    G::sync();
    cluster_sync_all();
    const uint32_t lead = peer_addr(smem_addr(xC), 0u);
#pragma unroll
    for (int k = 0; k < kViewAhead; ++k) {
      const int t = vt0 + k * G::kThreads + tid;
      if (t < vt1) red_add_peer(lead + 4u * (uint32_t)coarse_bin(vu[k]), 1u);
    }
    for (int t = vt0 + kViewAhead * G::kThreads + tid; t < vt1; t += G::kThreads)
      red_add_peer(lead + 4u * (uint32_t)coarse_bin(__ldg(reinterpret_cast<const unsigned int*>(row) +
                                                          a + (int64_t)t * p.s)),
                   1u);
    G::sync();
    cluster_sync_all();
    reinterpret_cast<uint4*>(sum)[tid] = ld_peer4(lead + 16u * (uint32_t)tid);
    static_assert(kCoarseBins == 4 * kClusterThreads, "one 4-bin vector per thread");
    G::sync();
    if (copy_late && tid == 0 && nb > 0)
      bulk_copy_g2s(smem_addr(stage), src, (uint32_t)nb * 4u, bar);
    view_cutoffs<G>(p, sum, sc, sl);
  } else if (!guess && !direct) {
    clear_hist<G>(sum, kCoarseBins);
    G::sync();
#pragma unroll
    for (int k = 0; k < kViewAhead; ++k) {
      const int t = k * G::kThreads + tid;
      if (t < vsize) {
        const uint32_t u =
            sampled ? vu[k] : __ldg(reinterpret_cast<const unsigned int*>(row) + a + (int64_t)t * p.s);
        atomicAdd(&sum[coarse_bin(u)], 1u);
      }
    }
    for (int t = kViewAhead * G::kThreads + tid; t < vsize; t += G::kThreads)
      atomicAdd(&sum[coarse_bin(__ldg(reinterpret_cast<const unsigned int*>(row) + a +
                                      (int64_t)t * p.s))],
                1u);
    G::sync();
    if (copy_late && tid == 0 && nb > 0)
      bulk_copy_g2s(smem_addr(stage), src, (uint32_t)nb * 4u, bar);
    view_cutoffs<G>(p, sum, sc, sl);
  }
  uint32_t T0 = sl.T0, T1 = sl.T1;
  if (guess || !(p.dual && T1 > T0)) T1 = T0;
  const int tau0 = sl.tau0, tau1 = guess ? -1 : sl.tau1;
  // One thread polls the copy's barrier; the rest wait at the CTA barrier.
  if (tid == 0 && nb > 0 && !mbar_wait_bounded(bar)) cs.timed_out = 1;
  G::sync();
  const uint4* st4 = reinterpret_cast<const uint4*>(stage);
  const int nv4 = (n + 3) >> 2;
  const int nh4 = (held + 3) >> 2;  // vectors held in shared memory
  // Scores 4t .. 4t+3 of the segment (positions >= n are junk for the caller
  // to mask): from shared memory below `held`, else from global memory.
  auto seg_vec = [&](int t) -> uint4 {
    if (t < nh4) return st4[t];
    if (bulk) return ldg_v4(src + 4 * t);
    uint4 v;
    v.x = 4 * t < n ? ld_stream1(src + 4 * t) : 0u;
    v.y = 4 * t + 1 < n ? ld_stream1(src + 4 * t + 1) : 0u;
    v.z = 4 * t + 2 < n ? ld_stream1(src + 4 * t + 2) : 0u;
    v.w = 4 * t + 3 < n ? ld_stream1(src + 4 * t + 3) : 0u;
    return v;
  };

  // ---- Phase 2 over the resident segment (one pass) ----
  // Both classes are counted per thread; every admitted key (d <= T1) and its
  // position go to the warp's region at a rank taken from a ballot, so the
  // pass needs no atomics.
  if (!direct) {
    // one ballot per score: every admitted key (d <= T1) and its position go
    // to the warp's region; its class (A: d <= T0) follows from the key.
    uint32_t wc = 0u;   // warp-uniform: admitted keys this warp found
    uint32_t ca = 0u;   // this lane's class-A keys
    uint32_t* wk = keys + warp * kRegionCap;
    uint16_t* wp = pos + warp * kRegionCap;
    // Called by whole warps; `ok` false for vectors past the segment.  A
    // warp whose 32 vectors hold no admissible score skips the per-score
    // ballots.
    const Screen scr1(T1);
    uint32_t kmn = 0xFFFFFFFFu;  // this lane's smallest admitted key
    auto classify = [&](const uint4& v, int t, bool ok) {
      if (__ballot_sync(kFull, ok && scr1.any(v)) == 0u) return;
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t d = desc_key(u[e]);
        const bool adm = ok && 4 * t + e < n && d <= T1;
        ca += (adm && d <= T0) ? 1u : 0u;
        if (adm) kmn = min(kmn, d);
        const uint32_t bal = __ballot_sync(kFull, adm);
        if (bal != 0u) {
          const uint32_t rk = wc + (uint32_t)__popc(bal & lt);
          if (adm && rk < (uint32_t)kRegionCap) {
            wk[rk] = d;
            wp[rk] = (uint16_t)(4 * t + e);
          }
          wc += (uint32_t)__popc(bal);
        }
      }
    };
    const uint4 none = make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
    const int nh4r = (nh4 + 31) & ~31;
    {
      // The part held in shared memory: the indices of vectors with an
      // admissible score go to a per-warp stack (in the private histogram,
      // unused until the selection), and each 32 of them are classified with
      // every lane busy instead of every vector step running the per-score
      // work for the few lanes that have any.
      uint32_t* wstack = hist + warp * 128;  // depth < 64
      uint32_t qn = 0u;                      // warp-uniform
      for (int t = tid; t < nh4r; t += G::kThreads) {
        const bool adm = t < nh4 && scr1.any(st4[t]);
        const uint32_t bal = __ballot_sync(kFull, adm);
        if (adm) wstack[qn + (uint32_t)__popc(bal & lt)] = (uint32_t)t;
        qn += (uint32_t)__popc(bal);
        if (qn >= 32u) {
          __syncwarp();
          const uint32_t tt = wstack[qn - 32u + (uint32_t)lane];
          __syncwarp();  // read before later pushes reuse the slots
          qn -= 32u;
          classify(st4[tt], (int)tt, true);
        }
      }
      if (qn > 0u) {
        __syncwarp();
        const bool has = (uint32_t)lane < qn;
        const uint32_t tt = has ? wstack[lane] : 0u;
        classify(has ? st4[tt] : none, (int)tt, has);
      }
    }
    // the part read from global memory: four vectors per thread in flight
    const int ntail = nv4 - nh4;
    const int ntr = (ntail + 31) & ~31;
    for (int b0 = 0; b0 < ntr; b0 += 4 * G::kThreads) {
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = b0 + k * G::kThreads + tid;
        v[k] = j < ntail ? seg_vec(nh4 + j) : none;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = b0 + k * G::kThreads + tid;
        if (b0 + k * G::kThreads + 32 * warp < ntr) classify(v[k], nh4 + j, j < ntail);
      }
    }
    ca = __reduce_add_sync(kFull, ca);
    kmn = __reduce_min_sync(kFull, kmn);
    if (lane == 0) {
      cs.wcnt[warp] = wc;
      atomicAdd(&cs.cnt_a, ca);
      atomicAdd(&cs.cnt_b, wc - ca);
      if (kmn != 0xFFFFFFFFu) atomicMin(&cs.kmin, kmn);
    }
  } else if (lane == 0) {
    cs.wcnt[warp] = 0u;
  }
  G::sync();
  cluster_sync_all();  // step 0: counts and key regions published

  // Certification over the cluster (eq. 27) and the layout of the merged
  // list: sub-list 16 j + w is warp w's region in CTA j, and h256[16 j + w]
  // its offset.  One warp issues every peer load at once.
  if (warp == 0) {
    uint32_t ca = 0u, cb = 0u, km = 0xFFFFFFFFu;
    if (lane < P) {
      ca = ld_peer(peer_addr(smem_addr(&cs.cnt_a), (uint32_t)lane));
      cb = ld_peer(peer_addr(smem_addr(&cs.cnt_b), (uint32_t)lane));
      km = ld_peer(peer_addr(smem_addr(&cs.kmin), (uint32_t)lane));
    }
    km = __reduce_min_sync(kFull, km);
    // 16 sub-lists per CTA, kSub per lane: 16 * kClusterMaxSplits in all
    constexpr int kSub = 16 * kClusterMaxSplits / 32;
    uint32_t c[kSub];
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
      const int rr = kSub * lane + i, j = rr >> 4, w = rr & 15;
      c[i] = j < P ? ld_peer(peer_addr(smem_addr(&cs.wcnt[w]), (uint32_t)j)) : 0u;
    }
    ca = __reduce_add_sync(kFull, ca);
    cb = __reduce_add_sync(kFull, cb);
    bool over = false;
    uint32_t s4 = 0u;
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
      over = over || c[i] > (uint32_t)kRegionCap;
      s4 += c[i];
    }
    uint32_t incl = s4;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t run = incl - s4;
#pragma unroll
    for (int i = 0; i < kSub; ++i) {
      h256[kSub * lane + i] = run;
      run += c[i];
    }
    over = __any_sync(kFull, over);
    if (lane == 0) {
      sl.c0 = (int)ca;
      sl.c1 = (int)cb;
      sc.bcast = over ? 1 : 0;
      sc.bcast2 = (int32_t)km;  // smallest admitted key of the row
    }
  }
  G::sync();
  const uint32_t C0 = (uint32_t)sl.c0, CB = (uint32_t)sl.c1;
  int route;
  bool recover;
  if (direct) {
    route = EXACT_TOPK_ROUTE_DIRECT_EXACT;
    recover = true;
  } else if (guess) {
    recover = C0 < (uint32_t)K;
    route = recover ? EXACT_TOPK_ROUTE_GUESS_EXACT : EXACT_TOPK_ROUTE_GUESS;
  } else if (C0 >= (uint32_t)K) {
    route = EXACT_TOPK_ROUTE_PRIMARY;
    recover = false;
  } else if (p.dual) {
    recover = C0 + CB < (uint32_t)K;
    route = recover ? EXACT_TOPK_ROUTE_EXACT_AFTER_BAND : EXACT_TOPK_ROUTE_BAND;
  } else {
    route = EXACT_TOPK_ROUTE_EXACT_NO_BAND;
    recover = true;
  }
  const bool band_tried = !direct && !guess && p.dual && C0 < (uint32_t)K;
  const int c0_trace = direct ? -1 : (int)C0;
  const int c1_trace = band_tried ? (int)(C0 + CB) : -1;

  KeyBand F;
  uint32_t k = (uint32_t)K;
  int tstar = -1, e0 = 0, q0n = 0;
  Cut cut{0, 0u, 0u, false};
  // every admitted key is gathered; the selection ignores keys above F.hi
  const uint32_t nfront = C0 + CB;
  const bool list_path = !recover && sc.bcast == 0 && nfront <= kMergeCap;
  if (!recover) {
    const bool with_b = route == EXACT_TOPK_ROUTE_BAND;
    F.has_lo = false;
    F.lo = 0u;
    F.hi = with_b ? T1 : T0;
    q0n = with_b ? (int)(C0 + CB) : (int)C0;
  }
  if (list_path) {
    // Merge every CTA's regions (independent DSMEM loads), then select the
    // K-th smallest frontier key locally: commit the keys below it and fill
    // the rest from its ties (eqs. 22-25 reach the same threshold).
    const uint32_t total = nfront;
    // Warp w copies the regions of warp w in every CTA: consecutive keys of
    // one peer region per request, all of a warp's requests in flight together.
    const uint32_t kb = smem_addr(keys);
    constexpr int kGroup = 4;  // CTAs whose regions are in flight together
    for (int j0 = 0; j0 < P; j0 += kGroup) {
      uint32_t vv[kGroup][4];
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int j = j0 + g;
#pragma unroll
        for (int x = 0; x < 4; ++x) vv[g][x] = 0u;
        if (j < P) {
          const int rr = 16 * j + warp;
          const uint32_t beg = h256[rr], end = rr + 1 < 16 * P ? h256[rr + 1] : total;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint32_t e = (uint32_t)lane + 32u * x;
            if (beg + e < end)
              vv[g][x] =
                  ld_peer(peer_addr(kb + 4u * ((uint32_t)warp * kRegionCap + e), (uint32_t)j));
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kGroup; ++g) {
        const int j = j0 + g;
        if (j < P) {
          const int rr = 16 * j + warp;
          const uint32_t beg = h256[rr], end = rr + 1 < 16 * P ? h256[rr + 1] : total;
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint32_t e = (uint32_t)lane + 32u * x;
            if (beg + e < end) sumx[beg + e] = vv[g][x];
          }
        }
      }
    }
    G::sync();
    uint32_t below;
    bool bad = false;
    // every gathered key lies in [smallest admitted key, F.hi] or above F.hi
    const uint32_t kmin_row = (uint32_t)sc.bcast2;
    const uint32_t vstar = small_select<G>(sumx, total, F.hi, k, hist, sc, below, bad,
                                           kmin_row <= F.hi, kmin_row);
    cut.bad = bad;
    cut.commit_below = vstar;
    cut.tie_key = vstar;
    cut.ties = k - below;
  } else if (!recover) {
    const uint32_t kmin_row = (uint32_t)sc.bcast2;  // smallest admitted key of the row
    cut = cluster_select<G>(seg_vec, n, F, k, xA, xC, sum, sc, P, kmin_row <= F.hi ? kmin_row : 0u);
  } else {
    // Exact coarse recovery (eq. 20) over the resident row: coarse histogram,
    // tau* = min{b : C(b) >= K}, E0 = {c < tau*}, Q0 = {c == tau*}.
    clear_hist<G>(xA, kCoarseBins);
    G::sync();
    {
      RunHist rh;
      for (int t = tid; t < nv4; t += G::kThreads) {
        const uint4 v = seg_vec(t);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * t + e < n) rh.add(xA, (uint32_t)coarse_bin(u[e]));
      }
      rh.flush(xA);
    }
    G::sync();
    cluster_sync_all();
    cluster_hist_sum<G>(xA, sum, kCoarseBins, P);
    find_boundaries<G>(sum, sc, kCoarseBins, 1, (uint32_t)K, 0u);
    tstar = sc.res_bin[0];
    e0 = (int)sc.res_below[0];
    q0n = (int)sc.res_cnt[0];
    exact_cutoffs<G>(sl, tstar < 0 ? 0 : tstar);
    F.has_lo = tstar > 0;
    F.lo = sl.T0;
    F.hi = sl.T1;
    k = (uint32_t)(K - e0);
    if (tstar < 0)
      cut.bad = true;
    else
      cut = cluster_select<G>(seg_vec, n, F, k, xC, xA, sum, sc, P, 0u);
  }
  G::sync();  // every thread holds the cut before the commit reuses the scratch

  // ---- commit ----
  const uint32_t a_out = peer_addr(smem_addr(&cs.n_out), 0u);
  const uint32_t a_keep = peer_addr(smem_addr(&cs.n_keep), 0u);
  if (list_path) {
    // candidates: this CTA's own admitted entries (regions), frontier keys only
    // candidates: each warp visits its own region (this CTA's admitted
    // entries), frontier keys only
    const uint32_t cw = cs.wcnt[warp];  // <= kRegionCap on this path
    const uint32_t hiF = F.hi;
    const uint32_t* wk = keys + warp * kRegionCap;
    const uint16_t* wp = pos + warp * kRegionCap;
    auto visit = [&](auto&& fn) {
      for (uint32_t i = lane; i < cw; i += 32) {
        const uint32_t d = wk[i];
        if (d <= hiF) fn(d, false, lo + (int32_t)wp[i]);
      }
    };
    cluster_commit<G>(visit, cut.commit_below, cut.tie_key, cut.ties, cut.bad, a_out, a_keep, sc,
                      out_row, K);
  } else {
    const KeyBand FF = F;
    auto visit = [&](auto&& fn) {
      for (int t = tid; t < nv4; t += G::kThreads) {
        const uint4 v = seg_vec(t);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t d = desc_key(u[e]);
          if (4 * t + e < n && (FF.below(d) || FF.in(d))) fn(d, FF.below(d), lo + 4 * t + e);
        }
      }
    };
    cluster_commit<G>(visit, cut.commit_below, cut.tie_key, cut.ties, cut.bad, a_out, a_keep, sc,
                      out_row, K);
  }
  G::sync();
  cluster_sync_all();  // every slot written; no CTA reads a peer after this

  if (q == 0) {
    const bool fill_ok = cs.n_out == (uint32_t)K - cut.ties && cs.n_keep >= cut.ties;
    if (cut.bad || !fill_ok) {
      for (int t = tid; t < K; t += G::kThreads) out_row[t] = -1;
      if (tid == 0) flag_status(p.counters, 1);
    }
    if (tid == 0)
      write_trace(p, r, route, direct ? -1 : tau0, direct ? -1 : tau1, c0_trace, c1_trace, tstar,
                  e0, q0n);
  }
  if (tid == 0 && cs.timed_out) flag_status(p.counters, 4);
}

// ----------------------------------------------------------------------------
// Streaming floor (measurement)
// ----------------------------------------------------------------------------

// Reads the valid prefix of every live row exactly once (P CTAs per row, the
// segments of segment_bounds, 256-bit loads with four in flight per thread)
// and writes one checksum word per CTA: the time a kernel needs to read a
// workload's algorithmic bytes in this launch shape, with nothing else to do.
constexpr int kFloorThreads = 512;

__global__ void __launch_bounds__(kFloorThreads) stream_floor_kernel(const float* logits,
                                                                     int64_t pitch, int N,
                                                                     int M_cap, const int32_t* ke,
                                                                     uint32_t* out) {
  const int r = blockIdx.y, P = gridDim.x, q = blockIdx.x;
  if (r >= M_cap) return;
  int L = ke[r];
  L = L < 0 ? 0 : (L > N ? N : L);
  int lo, hi;
  segment_bounds(L, P, q, lo, hi);
  const float* row = logits + (int64_t)r * pitch;
  uint32_t acc = 0u;
  if (lo < hi) {
    const Span sp = aligned_span(row, lo, hi);
    const int tid = threadIdx.x;
    const int head = sp.a0 - lo, tail = hi - sp.a_end;
    if (tid < head + tail) acc ^= ld_stream1(row + (tid < head ? lo + tid : sp.a_end + (tid - head)));
    const float* body = row + sp.a0;
    for (int v0 = 0; v0 < sp.nvec; v0 += 4 * kFloorThreads) {
      uint32_t x[4][8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = v0 + k * kFloorThreads + tid;
        if (v < sp.nvec) {
          ld_stream8(body + 8 * v, x[k]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[k][e] = 0u;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc ^= x[k][e];
    }
  }
  acc = __reduce_xor_sync(kFull, acc);
  __shared__ uint32_t wx[kFloorThreads / 32];
  if ((threadIdx.x & 31) == 0) wx[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0u;
    for (int w = 0; w < kFloorThreads / 32; ++w) t ^= wx[w];
    out[(int64_t)r * P + q] = t;
  }
}

// ----------------------------------------------------------------------------
// Heavy rows of the persistent kernel
// ----------------------------------------------------------------------------
//
// Rows whose Phase 1 predicts a frontier far beyond on-chip capacity (a tie
// group or a constant row admitted whole, the |Q0| = L worst case of section
// 4.4) are set aside by the persistent CTA that claimed them and finished in
// its epilogue, after its other rows, without materializing the frontier: the
// counts of eqs. 16-19 and the exact coarse recovery of eq. 20 when they fall
// short run as passes over the row itself, and so do the digit rounds of eqs.
// 22-25 until the keys left in play fit the on-chip frontier or are all equal
// (eq. 25's ties).  The routes and trace fields are those of the frontier
// method.

// Count, extremes and their multiplicities of a set of keys, and how many of
// them a histogram holds.
struct RowStats {
  uint32_t cnt, kmin, kmax, nmin, nmax, nhist;
};

// A digit histogram of the keys in [hlo, ...) of a set: digit (d - hlo) >> shift
// over nbins bins.
struct DigitHist {
  uint64_t hlo;
  int shift, nbins;
};

// Digit histogram over the keys of coarse bin tau, [cutoff(tau - 1) + 1, T]
// with T = cutoff(tau): 11 bits of the bin's key range.  Whole group; the
// result is valid for every thread.
template <class G>
__device__ DigitHist bin_digits(int tau, uint32_t T, GroupScratch& sc) {
  G::sync();  // the scratch is free
  if (G::rank() < 32) {
    const uint32_t lo = tau > 0 ? cutoff_fast_warp(tau - 1) + 1u : 0u;
    if (G::rank() == 0) sc.bcast2 = (int32_t)lo;
  }
  G::sync();
  DigitHist h;
  h.hlo = (uint32_t)sc.bcast2;
  const uint64_t w = (uint64_t)T + 1u - h.hlo;  // >= 1
  const int bits = 64 - __clzll((long long)(w - 1u | 1u));
  h.shift = bits > 11 ? bits - 11 : 0;
  h.nbins = (int)((((w - 1u) >> h.shift) + 1u + 127u) & ~127ull);
  return h;
}

// Count, smallest and largest of the keys d <= T in [qlo, qhi) of the row and
// how many keys equal each, and (hist not null) the digit histogram `dh` of
// those at or above dh.hlo from a clear one; block-wide results, valid for
// every thread on return.
template <class G>
__device__ void row_pass(const float* row, int L, uint32_t T, uint64_t qlo, uint64_t qhi,
                         const DigitHist& dh, uint32_t* hist, GroupScratch& sc, RowStats& st) {
  G::sync();  // hist and the scratch are free
  if (hist != nullptr) clear_hist<G>(hist, dh.nbins);
  if (G::rank() == 0) {
    sc.bcast = 0;
    sc.res_cnt[0] = 0u;
    sc.res_cnt[1] = 0u;
    sc.res_below[0] = 0u;
    prefetch_row_l2(row, L);
  }
  G::sync();
  uint32_t c = 0u, mn = 0xFFFFFFFFu, mx = 0u, nmn = 0u, nmx = 0u, nh = 0u;
  scan_key_hist<G>(row, L, T, qlo, qhi, dh.hlo, dh.shift, hist, c, mn, mx, nmn, nmx, nh);
  c = __reduce_add_sync(kFull, c);
  nh = __reduce_add_sync(kFull, nh);
  if ((G::rank() & 31) == 0) {
    if (c) atomicAdd(&sc.bcast, (int)c);
    if (nh) atomicAdd(&sc.res_below[0], nh);
  }
  uint32_t kmin, kmax;
  block_min_max<G>(mn, mx, sc, kmin, kmax);  // ends with a group barrier
  const uint32_t a = __reduce_add_sync(kFull, mn == kmin ? nmn : 0u);
  const uint32_t b = __reduce_add_sync(kFull, mx == kmax ? nmx : 0u);
  if ((G::rank() & 31) == 0) {
    if (a) atomicAdd(&sc.res_cnt[0], a);
    if (b) atomicAdd(&sc.res_cnt[1], b);
  }
  G::sync();
  st = RowStats{(uint32_t)sc.bcast, kmin, kmax, sc.res_cnt[0], sc.res_cnt[1], sc.res_below[0]};
}

// Final pass of the heavy-row selection when the keys in play fit the shared
// frontier: every key d <= T below qlo goes to the output, every key in [qlo,
// qhi) to the frontier (positions through sl.n_keep).  Ends with a group
// barrier.
template <class G>
__device__ void collect_pass(const float* row, int L, uint32_t T, uint64_t qlo, uint64_t qhi,
                             const Frontier& F, Slot& sl, int32_t* out_row, int K) {
  G::sync();  // the frontier is free
  if (G::rank() == 0) {
    sl.n_keep = 0u;
    prefetch_row_l2(row, L);
  }
  G::sync();
  auto step = [&](const uint32_t* x, int i0, int nvalid) {
    uint32_t cm = 0u, qm = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t d = desc_key(x[e]);
      const bool ok = e < nvalid && d <= T;
      if (ok && (uint64_t)d < qlo)
        cm |= 1u << e;
      else if (ok && (uint64_t)d < qhi)
        qm |= 1u << e;
    }
    if (__ballot_sync(kFull, cm != 0u) != 0u) commit_mask(cm, i0, &sl.n_out, out_row, K);
    if (__ballot_sync(kFull, qm != 0u) != 0u) {
      uint32_t tot;
      const uint32_t ex = warp_excl_scan((uint32_t)__popc(qm), tot);
      uint32_t base = 0u;
      if ((threadIdx.x & 31) == 0) base = atomicAdd(&sl.n_keep, tot);
      uint32_t pos = __shfl_sync(kFull, base, 0) + ex;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (qm & (1u << e)) {
          if (pos < F.cap) F.s[pos] = make_uint2((uint32_t)(i0 + e), desc_key(x[e]));
          ++pos;
        }
      }
    }
  };
  visit_row<G>(row, L, step, []() { return false; });
  G::sync();
}

// 11 digit bits over the keys [lo, hi].
__device__ __forceinline__ DigitHist digits_over(uint64_t lo, uint64_t hi) {
  DigitHist h;
  h.hlo = lo;
  const uint64_t w = hi + 1u - lo;  // >= 1
  const int bits = 64 - __clzll((long long)(w - 1u | 1u));
  h.shift = bits > 11 ? bits - 11 : 0;
  h.nbins = (int)((((w - 1u) >> h.shift) + 1u + 127u) & ~127ull);
  return h;
}

// Phase 3 over the row itself (eqs. 22-25): the k smallest of the keys in
// play, the keys d <= T in [st.kmin, st.kmax] that `st` describes, every key
// d <= T below them taken whole.  Each step first tries to close the
// selection from the counts alone: k or more keys equal the smallest (k
// ties, eq. 25), or fewer than k lie below the largest (all of them, then
// ties at the largest); both end with one commit pass.  Keys in play that fit
// the shared frontier are collected by one pass and refined on chip.
// Otherwise a digit histogram of the keys in play (the one the last pass
// built when `pre`, over [h.hlo, ...), else one more pass over their measured
// range) gives the bucket holding the k-th key; the bucket closes the quota,
// is collected, or becomes the keys in play, measured and histogrammed by one
// pass.  Returns false on inconsistent counts.
template <class G>
__device__ bool heavy_select(const float* row, int L, uint32_t T, uint32_t k, RowStats st,
                             DigitHist h, bool pre, uint32_t* hist, const Frontier& F,
                             GroupScratch& sc, Slot& sl, int32_t* out_row, int K,
                             uint32_t* scratch, uint32_t scap) {
  for (int round = 0; round < 8; ++round) {
    if (k == 0u || st.cnt < k || st.kmin > st.kmax) break;  // inconsistent counts
    if (st.nmin >= k) {
      scan_commit<G>(row, L, T, 0u, st.kmin, st.kmin, k, sl, out_row, K);
      return true;
    }
    if (st.cnt - st.nmax < k) {
      scan_commit<G>(row, L, T, 0u, st.kmax, st.kmax, k - (st.cnt - st.nmax), sl, out_row, K);
      return true;
    }
    if (st.cnt <= F.cap) {
      collect_pass<G>(row, L, T, st.kmin, (uint64_t)st.kmax + 1u, F, sl, out_row, K);
      refine<G>(F, st.cnt, k, hist, sc, sl, out_row, K, scratch, scap);
      return true;
    }
    const uint32_t under = pre ? st.cnt - st.nhist : 0u;  // keys in play below the histogram
    if (!pre || under >= k) {
      h = digits_over(st.kmin, st.kmax);
      row_pass<G>(row, L, T, st.kmin, (uint64_t)st.kmax + 1u, h, hist, sc, st);
      pre = true;
      continue;
    }
    find_boundaries<G>(hist, sc, h.nbins, 1, k - under, 0u);
    const int b = sc.res_bin[0];
    if (b < 0) break;
    const uint32_t below = sc.res_below[0] + under, bc = sc.res_cnt[0];
    const uint64_t qlo = h.hlo + ((uint64_t)b << h.shift);
    uint64_t qhi = qlo + ((uint64_t)1 << h.shift);
    if (qhi > (uint64_t)st.kmax + 1u) qhi = (uint64_t)st.kmax + 1u;
    if (below + bc == k) {
      // the bucket closes the quota: everything below its top
      scan_commit<G>(row, L, T, 0u, qhi, 0u, 0u, sl, out_row, K);
      return true;
    }
    k -= below;
    if (bc <= F.cap) {
      collect_pass<G>(row, L, T, qlo, qhi, F, sl, out_row, K);
      refine<G>(F, bc, k, hist, sc, sl, out_row, K, scratch, scap);
      return true;
    }
    // the bucket becomes the keys in play: its counts and next digit in one pass
    h = digits_over(qlo, qhi - 1u);
    row_pass<G>(row, L, T, qlo, qhi, h, hist, sc, st);
    pre = true;
  }
  return false;
}

template <class G>
__device__ void heavy_row(const Params& p, const int32_t* rec, uint32_t* hist, GroupScratch& sc,
                          Slot& sl, const Frontier& F, uint32_t* scratch, uint32_t scap) {
  const int r = rec[0], L = rec[1];
  const uint32_t T0 = (uint32_t)rec[2], T1 = (uint32_t)rec[3];
  const int tau0 = rec[4], tau1 = rec[5];
  const int K = p.K;
  const float* row = p.logits + (int64_t)r * p.pitch;
  int32_t* out_row = p.out + (int64_t)r * K;
  if (G::rank() == 0) {
    sl.n_out = 0u;
    sl.n_keep = 0u;
  }
  // Phase 2 counts (eqs. 16-19) with the range of the admitted keys and a
  // digit histogram of the keys in the cutoff's own coarse bin, where a heavy
  // row's mass sits
  RowStats st;
  DigitHist dh = bin_digits<G>(tau0, T0, sc);
  row_pass<G>(row, L, T0, 0u, (uint64_t)T0 + 1u, dh, hist, sc, st);
  const uint32_t c0 = st.cnt;
  int route, c1 = -1, tstar = -1, e0 = 0, q0;
  uint32_t T = T0;
  bool ok = true;
  if (c0 >= (uint32_t)K) {
    route = EXACT_TOPK_ROUTE_PRIMARY;
    q0 = (int)c0;
  } else {
    route = EXACT_TOPK_ROUTE_EXACT_NO_BAND;
    q0 = 0;
    if (p.dual) {
      dh = bin_digits<G>(tau1, T1, sc);
      row_pass<G>(row, L, T1, 0u, (uint64_t)T1 + 1u, dh, hist, sc, st);
      c1 = (int)st.cnt;  // band rescue: C(tau1)
      route = c1 >= K ? EXACT_TOPK_ROUTE_BAND : EXACT_TOPK_ROUTE_EXACT_AFTER_BAND;
      T = T1;
      q0 = c1;
    }
    if (route != EXACT_TOPK_ROUTE_BAND) {
      // exact coarse recovery (eq. 20): tau* = min{b : C(b) >= K}; the keys of
      // bins below tau* (E0) are committed by the final pass, Q0 = bin tau*
      G::sync();
      clear_hist<G>(hist, 2048);
      if (G::rank() == 0) prefetch_row_l2(row, L);
      G::sync();
      scan_coarse_hist<G>(row, 0, L, hist);
      G::sync();
      find_boundaries<G>(hist, sc, 2048, 1, (uint32_t)K, 0u);
      tstar = sc.res_bin[0];
      e0 = (int)sc.res_below[0];
      q0 = (int)sc.res_cnt[0];
      ok = tstar >= 0;
      exact_cutoffs<G>(sl, ok ? tstar : 0);
      T = sl.T1;
      const uint32_t lo = tstar > 0 ? sl.T0 + 1u : 0u;
      dh = digits_over(lo, T);
      row_pass<G>(row, L, T, lo, (uint64_t)T + 1u, dh, hist, sc, st);
    }
  }
  if (ok)
    heavy_select<G>(row, L, T, (uint32_t)(K - e0), st, dh, true, hist, F, sc, sl, out_row, K,
                    scratch, scap);
  finish_row<G>(p, sl, out_row);
  if (G::rank() == 0) write_trace(p, r, route, tau0, tau1, (int)c0, c1, tstar, e0, q0);
}

// Out of line, with its shared-memory views rebuilt here: nothing of the
// epilogue stays live through the row loop.
__device__ __noinline__ void finish_deferred(const Params& p) {
  using G = CtaGroup<kPersistentThreads>;
  unsigned char* sm = smem_base();
  constexpr SmemLayout lay = smem_layout(EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, kPersistentCap);
  const uint32_t* own = reinterpret_cast<const uint32_t*>(sm + lay.own);
  uint32_t* hist = reinterpret_cast<uint32_t*>(sm + lay.hist);
  GroupScratch& sc = *reinterpret_cast<GroupScratch*>(sm + lay.scratch);
  Slot& sl = *reinterpret_cast<Slot*>(sm + lay.slots);
  const Frontier F{reinterpret_cast<uint2*>(sm + lay.frontier), (uint32_t)kPersistentCap, nullptr,
                   (uint32_t)kPersistentCap};
  uint32_t* scratch = reinterpret_cast<uint32_t*>(sm + lay.queues);
  const uint32_t n = own[0];
  for (uint32_t j = 0; j < n; ++j) {
    heavy_row<G>(p, p.defer + 8 * (int64_t)own[1 + j], hist, sc, sl, F, scratch,
                 (uint32_t)(G::kWarps * kQueueWords));
    __syncthreads();
  }
}

// Kernel attributes are set once per (device, kernel); later launches, which
// may be inside a stream capture, only launch.
constexpr int kMaxDevices = 64;
volatile int g_attr_smem[kMaxDevices][5];

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
  // clusters of up to 16 CTAs (the portable limit is 8)
  if (family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  if (cached) g_attr_smem[dev][family] = (int)smem;
  return EXACT_TOPK_OK;
}

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (no link-time dependency on the driver library); null when unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// The persistent kernel's view map (Params::view_map): the scores of row z as
// lines of s, box {4, min(256, N / s), 1}.  Only when s and the row pitch are
// multiples of 4 scores (16-byte strides, 16-byte x coordinates a & ~3) and
// the base is 16-byte aligned; otherwise the kernel gathers with plain loads.
bool encode_view_map(Params& p) {
  if (p.s < 4 || (p.s & 3) != 0 || (p.pitch & 3) != 0 || p.N < p.s || p.M_cap < 1) return false;
  if ((reinterpret_cast<uintptr_t>(p.logits) & 15u) != 0u) return false;
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t lines = (cuuint64_t)(p.N / p.s);
  const cuuint32_t box = (cuuint32_t)(lines < 256u ? lines : 256u);
  const cuuint64_t dims[3] = {(cuuint64_t)p.s, lines, (cuuint64_t)p.M_cap};
  const cuuint64_t strides[2] = {(cuuint64_t)p.s * 4u, (cuuint64_t)p.pitch * 4u};
  const cuuint32_t boxdim[3] = {4u, box, 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  if (fn(&p.view_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3u, const_cast<float*>(p.logits), dims,
         strides, boxdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  p.view_box = (int32_t)box;
  return true;
}

}  // namespace

size_t shared_bytes(int family, int cap) {
  if (family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT) return cluster_layout().total;
  return smem_layout(family, cap).total;
}

int kernel_occupancy(int family, int device, int* ctas_per_sm) {
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  int rc = EXACT_TOPK_OK, n = 0;
  cudaError_t e = cudaSuccess;
  if (family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED) {
    (void)encode_tiled();  // resolved here, at planning time, not inside a capture
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
  } else if (family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT) {
    const size_t smem = shared_bytes(family, kClusterStage);
    rc = set_attrs(cluster_split_kernel, EXACT_TOPK_FAMILY_CLUSTER_SPLIT, smem);
    if (rc == EXACT_TOPK_OK)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, cluster_split_kernel, kClusterThreads,
                                                        smem);
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
  p.defer = plan.family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED && ws != nullptr
                ? reinterpret_cast<int32_t*>(ws + lay.defer_offset)
                : nullptr;
  p.prev = a.prev_topk;
  p.trace = a.trace;
  p.view_tma = 0;
  p.view_box = 0;
  memset(&p.view_map, 0, sizeof(p.view_map));
  if (plan.family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED && encode_view_map(p)) p.view_tma = 1;
  const size_t smem = shared_bytes(plan.family, plan.cand_capacity);
  int rc = EXACT_TOPK_OK;
  switch (plan.family) {
    case EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED:
      rc = set_attrs(persistent_sampled_kernel, EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, smem);
      if (rc != EXACT_TOPK_OK) return rc;
      persistent_sampled_kernel<<<plan.workers, kPersistentThreads, smem, stream>>>(p);
      // rows the persistent kernel deferred (predicted frontiers far beyond
      // on-chip capacity); exits at once when there are none

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
    case EXACT_TOPK_FAMILY_CLUSTER_SPLIT: {
      if (plan.splits < 1 || plan.splits > kClusterMaxSplits ||
          (int64_t)plan.splits * kClusterSegment < plan.max_kv_len)
        return EXACT_TOPK_ERR_BAD_PLAN;
      rc = set_attrs(cluster_split_kernel, EXACT_TOPK_FAMILY_CLUSTER_SPLIT, smem);
      if (rc != EXACT_TOPK_OK) return rc;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.num_rows, 1u);
      cfg.blockDim = dim3(kClusterThreads, 1u, 1u);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)plan.splits;
      attr[0].val.clusterDim.y = 1u;
      attr[0].val.clusterDim.z = 1u;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, cluster_split_kernel, p) != cudaSuccess)
        return EXACT_TOPK_ERR_CUDA;
      break;
    }
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
// Top-K: plugins whose host framework owns every device allocation, and
// latency-critical loops where cudaMalloc's implicit device synchronization is
// unacceptable.  For them this entry point runs the KV-split kernel with its
// counters and workspace carved out of one file-scope device array instead of
// caller-provided buffers.

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
  // Every argument check runs before anything is enqueued, so a rejected call
  // leaves the stream and the array untouched.
  rc = check_run(&plan, logits, ke, out, num_valid_rows, scratch, (size_t)plan.counter_bytes,
                 scratch + ctr_bytes, (size_t)plan.workspace_bytes, nullptr, nullptr);
  if (rc != EXACT_TOPK_OK) return rc;
  // The array keeps whatever the previous call left; the counters must start
  // at zero, so clear them on the stream (a memset, not an allocation).
  if (cudaMemsetAsync(scratch, 0, (size_t)plan.counter_bytes,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  return exact_topk_run(&plan, logits, ke, out, num_valid_rows, scratch,
                        (size_t)plan.counter_bytes, scratch + ctr_bytes,
                        (size_t)plan.workspace_bytes, nullptr, nullptr, stream);
}

extern "C" int exact_topk_stream_floor(const float* logits, int64_t num_rows, int64_t max_kv_len,
                                       int64_t row_pitch, const int32_t* ke, uint32_t* out,
                                       int splits, struct CUstream_st* stream) {
  using namespace etk;
  if (logits == nullptr || ke == nullptr || out == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  if (num_rows < 1 || num_rows > 65535 || max_kv_len < 1 || max_kv_len > EXACT_TOPK_MAX_N ||
      row_pitch < max_kv_len)
    return EXACT_TOPK_ERR_BAD_SHAPE;
  if (splits < 1 || splits > 1024) return EXACT_TOPK_ERR_BAD_PLAN;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0u ||
      (reinterpret_cast<uintptr_t>(ke) & 3u) != 0u ||
      (reinterpret_cast<uintptr_t>(out) & 3u) != 0u)
    return EXACT_TOPK_ERR_MISALIGNED;
  const dim3 grid((unsigned)splits, (unsigned)num_rows);
  stream_floor_kernel<<<grid, kFloorThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      logits, row_pitch, (int)max_kv_len, (int)num_rows, ke, out);
  return cudaGetLastError() == cudaSuccess ? EXACT_TOPK_OK : EXACT_TOPK_ERR_CUDA;
}
