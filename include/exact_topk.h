/*
 * exact_topk.h -- C ABI of the GB300 (sm_103a) exact row-wise FP32 Top-K library.
 *
 * Operation ("Sample-Guided Exact Top-K Selection for Long-Context Sparse
 * Attention", section 2.1 "Operator contract"; API of the HPC-Ops pull request
 * "feat(topk): add sample-verified exact Top-K", section "API"):
 *
 *   Given a float32 score matrix X[num_rows][row_pitch] whose row r is valid on
 *   [0, L_r) with L_r = clamp(ke[r], 0, max_kv_len), write out[r][0..K) for every
 *   live row r < M_live = *num_valid_rows:
 *     - L_r >  K: K distinct indices i in [0, L_r) such that no unselected valid
 *                 score exceeds a selected one (exactness criterion, section 6.1
 *                 eq. 30).  Among scores tied at the K-th rank any choice is
 *                 valid; the selected VALUES are unique.
 *     - L_r <= K: every valid index 0..L_r-1, and -1 in the remaining slots.
 *   Slot order within a row is unspecified.  Rows r >= M_live are not written.
 *   Scores are compared by their IEEE-754 total order: +-inf and subnormals are
 *   ordered numerically and -0 ranks just below +0.  NaN is outside the
 *   contract (section 2.1); it is never a fault: a NaN ranks by its bit
 *   pattern (positive NaN above +inf, negative NaN below -inf).
 *   Padded columns j >= L_r may hold anything, NaN included; they are never read
 *   as data.
 *
 * Method: the sample-guided three-phase scheme of sections 4.2-4.5 (fixed-stride
 * view and coarse boundary, fused complete-row certification and candidate
 * formation, band rescue, exact coarse recovery, 11+11+10 radix refinement),
 * executed by one of three kernel families chosen by a host planner
 * (section 5.5, "Shape-stable dispatch").
 *
 * Conventions for every entry point:
 *   - Return 0 on success or a negative exact_topk_status; on error nothing is
 *     launched and no buffer is touched.
 *   - Pointers named "device" must be device (or managed) memory of the current
 *     CUDA device; the library never dereferences them on the host.
 *   - The caller owns every buffer.  The library allocates no memory, never
 *     synchronizes, never reads device memory back to the host, and enqueues
 *     work only on the given stream, so a call can be captured in a CUDA graph
 *     (section 2.1, "Deployment requirements").  The first call on a device
 *     queries device attributes and sets kernel attributes: make it once
 *     before starting a stream capture.
 *   - Calls on the same buffers must not overlap in time on the GPU.
 */
#ifndef EXACT_TOPK_H_
#define EXACT_TOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t == struct CUstream_st* ; NULL = legacy default stream */

typedef enum exact_topk_status {
  EXACT_TOPK_OK = 0,
  EXACT_TOPK_ERR_NULL_POINTER = -1,     /* a required pointer is NULL */
  EXACT_TOPK_ERR_BAD_SHAPE = -2,        /* num_rows < 1, max_kv_len < 1, row_pitch < max_kv_len, or too large */
  EXACT_TOPK_ERR_BAD_K = -3,            /* top_k < 1 or above EXACT_TOPK_MAX_K */
  EXACT_TOPK_ERR_COUNTERS_TOO_SMALL = -4,
  EXACT_TOPK_ERR_WORKSPACE_TOO_SMALL = -5,
  EXACT_TOPK_ERR_MISALIGNED = -6,       /* logits/ke/out/counters/workspace not 4-byte aligned
                                           (counters and workspace must be 16-byte aligned) */
  EXACT_TOPK_ERR_BAD_PLAN = -7,         /* a plan field is out of range or inconsistent */
  EXACT_TOPK_ERR_CUDA = -8              /* a CUDA runtime call failed (device query or launch) */
} exact_topk_status;

#define EXACT_TOPK_MAX_K 16384
#define EXACT_TOPK_MAX_N 0x7FFFFFF0LL    /* row width and pitch must fit int32 indices */

typedef enum exact_topk_family {
  /* The planner's choice, from the row count M, width N and the device:
     - N < 16384: row-local exact when the rows fit one wave of its CTAs or
       N < 1024, persistent sampled otherwise;
     - M < SM count: cluster split when a row fits the shared memory of a
       cluster of 8 (N <= 8 * 16384) and the clusters fit about two waves
       (clusters of up to 16 CTAs, N <= 16 * 32768, on request only);
       otherwise the KV-split, unless it would give each row a single segment
       (persistent sampled then);
     - otherwise persistent sampled. */
  EXACT_TOPK_FAMILY_AUTO = 0,
  /* One CTA owns a row for all three phases; rows are claimed from a device
     queue in completion order (section 5.5, "Persistent sampled").  A row
     whose view predicts a frontier beyond four on-chip capacities (a tie
     group, a constant row: section 4.4's |Q0| = L case) is finished after the
     CTA's other rows by passes over the row itself, with the same routes and
     trace. */
  EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED = 1,
  /* P CTAs scan disjoint segments of one row; the last to arrive finishes the
     row (section 4.5 eqs. 26-27; section 5.5, "Sampled KV-split"). */
  EXACT_TOPK_FAMILY_KV_SPLIT = 2,
  /* One wide CTA per row takes the exact coarse route directly; short rows stay
     in registers (section 5.5, "Row-local exact"). */
  EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT = 3,
  /* The P CTAs of one thread-block cluster (P <= 16) split one row into
     segments of at most 32768 scores; each CTA holds up to 16384 of them in
     shared memory (a TMA bulk copy) and reads the rest of its segment from
     global memory after an L2 prefetch.  The merge of eq. 27 and every later
     step run on chip through distributed shared memory (the KV-split
     decomposition of section 4.5 for rows that fit a cluster). */
  EXACT_TOPK_FAMILY_CLUSTER_SPLIT = 4
} exact_topk_family;

/* Route codes written to the optional per-row trace (Table 2 of section 4.6,
   plus the pad route of section 2.1 and the optional guess source). */
typedef enum exact_topk_route {
  EXACT_TOPK_ROUTE_PAD = 0,              /* L <= K */
  EXACT_TOPK_ROUTE_PRIMARY = 1,          /* C(tau0) >= K */
  EXACT_TOPK_ROUTE_BAND = 2,             /* C(tau0) < K <= C(tau1) */
  EXACT_TOPK_ROUTE_EXACT_AFTER_BAND = 3, /* C(tau1) < K: exact coarse recovery */
  EXACT_TOPK_ROUTE_EXACT_NO_BAND = 4,    /* primary-only policy, C(tau0) < K */
  EXACT_TOPK_ROUTE_DIRECT_EXACT = 5,     /* view unusable or row-local family */
  EXACT_TOPK_ROUTE_GUESS = 6,            /* previous-step Top-K certified */
  EXACT_TOPK_ROUTE_GUESS_EXACT = 7       /* guess underfilled: exact coarse recovery */
} exact_topk_route;

/* Per-row trace record: EXACT_TOPK_TRACE_FIELDS int32 per row, -1 where a
   field is not computed on the row's route. */
#define EXACT_TOPK_TRACE_FIELDS 8
/* [0] route  [1] tau0 (or the guessed boundary)  [2] tau1  [3] C(tau0)
   [4] C(tau1) when the band was tried  [5] tau* (exact coarse boundary)
   [6] |E0|  [7] |Q0| */

/* Device facts the planner needs; filled by exact_topk_query_device. */
typedef struct exact_topk_device_info {
  int32_t sm_count;
  int32_t persistent_ctas_per_sm; /* resident CTAs/SM of the persistent sampled kernel */
  int32_t kvsplit_ctas_per_sm;    /* resident CTAs/SM of the KV-split kernel */
  int32_t rowlocal_ctas_per_sm;   /* resident CTAs/SM of the row-local exact kernel */
  int32_t cluster_ctas_per_sm;    /* resident CTAs/SM of the cluster split kernel */
} exact_topk_device_info;

/* Optional planner overrides: 0 (or -1 where noted) keeps the planner's choice. */
typedef struct exact_topk_plan_request {
  int32_t family;        /* exact_topk_family */
  int32_t stride;        /* view stride s: power of two in [2, 4096] */
  int32_t dual;          /* -1 planner, 0 primary-only, 1 primary + secondary boundary */
  int32_t splits;        /* segment count P: KV-split [1, 128]; cluster split [1, 16]
                            with P * 32768 >= max_kv_len */
  int32_t workers;       /* persistent / row-local grid size */
  int32_t rho0_num, rho0_den; /* primary retention margin rho (K~ = rho K), default 3/2 */
  int32_t rho1_num, rho1_den; /* secondary margin rho1, default 7/4 */
} exact_topk_plan_request;

/* A complete launch plan.  Fixed before capture from (num_rows, max_kv_len,
   row_pitch, top_k, device); live row count and lengths stay device inputs. */
typedef struct exact_topk_plan {
  int32_t family;
  int32_t stride;
  int32_t dual;
  int32_t splits;
  int32_t workers;
  int32_t threads;        /* CTA size */
  int32_t top_k;
  int32_t q0, q1;         /* sample ranks ceil(rho0 K / s), ceil(rho1 K / s) */
  int32_t rho0_num, rho0_den, rho1_num, rho1_den;
  int32_t cand_capacity;  /* on-chip frontier entries per CTA */
  int32_t sm_count;
  int32_t reserved;
  int64_t num_rows;       /* M_cap */
  int64_t max_kv_len;     /* N */
  int64_t row_pitch;      /* floats between row starts (>= N) */
  uint64_t counter_bytes;
  uint64_t workspace_bytes;
} exact_topk_plan;

/* Fills *info for CUDA device `device` (occupancy of each kernel family).
   Host only; no launch, no sync.  Errors: ERR_NULL_POINTER, ERR_CUDA. */
int exact_topk_query_device(int device, exact_topk_device_info* info);

/* The host planner (section 5.5, "Shape-stable dispatch"): picks the kernel
   family, view stride s, primary/secondary policy, split count P, worker count
   and the counter/workspace sizes.  Pure host logic; `request` may be NULL.
   Errors: ERR_NULL_POINTER, ERR_BAD_SHAPE, ERR_BAD_K, ERR_BAD_PLAN. */
int exact_topk_make_plan(int64_t num_rows, int64_t max_kv_len, int64_t row_pitch, int top_k,
                         const exact_topk_device_info* info, const exact_topk_plan_request* request,
                         exact_topk_plan* plan);

/* Sizes of the two caller-owned buffers for the current device's default plan
   (PR API, topk_filtered_workspace_size).  `top_k` is an addition to the PR's
   signature: the plan, and hence the sizes, depend on it.
   counters: zero-filled once by the caller before first use; every launch
             returns it to all-zero (section 5.5; PR "API").
   workspace: needs no initialization and may persist across graph replays.
   Errors: ERR_NULL_POINTER, ERR_BAD_SHAPE, ERR_BAD_K, ERR_CUDA. */
int exact_topk_workspace_size(int64_t num_rows, int64_t max_kv_len, int top_k,
                              size_t* counter_bytes, size_t* workspace_bytes);

/* Exact Top-K with the current device's default plan (row_pitch = max_kv_len).
 *   logits          device float32 [num_rows][max_kv_len], 4-byte aligned
 *                   (16-byte aligned rows enable 128-bit loads)
 *   ke              device int32 [num_rows]: valid lengths, clamped to [0, max_kv_len]
 *   out             device int32 [num_rows][top_k]
 *   num_valid_rows  device int32 [1]: M_live, clamped to [0, num_rows];
 *                   NULL means M_live = num_rows
 *   counters        device, >= counter_bytes, 16-byte aligned, all-zero on entry
 *   workspace       device, >= workspace_bytes, 16-byte aligned, contents ignored
 *   prev_topk       NULL, or device int32 [num_rows][top_k]: a previous step's
 *                   Top-K used as an optional proposal.  A row uses it only
 *                   when all K entries lie in [0, L_r); the proposal is certified
 *                   by the same complete-row count, so the result is exact
 *                   whatever it holds.
 *   stream          CUDA stream (NULL = legacy default stream)
 * Enqueues one kernel.  Errors: any exact_topk_status; ERR_CUDA if the launch fails. */
int exact_topk(const float* logits, int64_t num_rows, int64_t max_kv_len, const int32_t* ke,
               int32_t* out, const int32_t* num_valid_rows, int top_k, void* counters,
               size_t counter_bytes, void* workspace, size_t workspace_bytes,
               const int32_t* prev_topk, struct CUstream_st* stream);

/* Same as exact_topk with an explicit plan (from exact_topk_make_plan) and an
   optional per-row trace: `trace` is NULL or device int32
   [plan->num_rows][EXACT_TOPK_TRACE_FIELDS], written for live rows only. */
int exact_topk_run(const exact_topk_plan* plan, const float* logits, const int32_t* ke,
                   int32_t* out, const int32_t* num_valid_rows, void* counters,
                   size_t counter_bytes, void* workspace, size_t workspace_bytes,
                   const int32_t* prev_topk, int32_t* trace, struct CUstream_st* stream);

/* Allocation-free variant of exact_topk, for callers that cannot allocate
 * device memory where they need the selection: plugins and extensions whose
 * host framework owns every device allocation (and hands them only the
 * tensors of the operation), and latency-critical loops where cudaMalloc's
 * implicit device synchronization is not acceptable.  The paper has no
 * counterpart to this entry point.
 *
 * It always runs the KV-split kernel family (planned as for exact_topk with
 * the family fixed) and takes its counters and workspace from one static
 * device array of EXACT_TOPK_NOALLOC_SCRATCH_BYTES that every GPU using the
 * library holds until the process exits.  The caller still passes the scores,
 * lengths, live-row count and output, with the meaning, layout and alignment
 * rules of exact_topk; there is no guess source.
 *   - Shapes whose KV-split counters (rounded up to 256 bytes) plus workspace
 *     (about num_rows * max_kv_len * 8 bytes) exceed the array are rejected
 *     with EXACT_TOPK_ERR_WORKSPACE_TOO_SMALL.  Every argument is checked
 *     before anything is enqueued: a rejected call launches nothing.
 *   - The first call on a device resolves the array's device address and the
 *     device's attributes; later calls on that device reuse them.  The kernel's
 *     attributes are set at the device's first launch of the KV-split family,
 *     by this or any other entry point.
 *   - Each call enqueues a memset of the counter region and one kernel on
 *     `stream`; it calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents: calls that overlap on the GPU (other streams, other
 *     host threads) race and must be serialized by the caller.
 *   - The sticky device-side status word (set when an internal consistency
 *     guard trips, which valid inputs never do) lives in that array and is
 *     cleared by the next call: this entry point cannot report it.
 * Errors: as exact_topk. */
#define EXACT_TOPK_NOALLOC_SCRATCH_BYTES (64u << 20)
int exact_topk_kv_split_noalloc(const float* logits, int64_t num_rows, int64_t max_kv_len,
                                const int32_t* ke, int32_t* out, const int32_t* num_valid_rows,
                                int top_k, struct CUstream_st* stream);

/* Measurement utility, not part of the selection: reads the valid prefix
 * [0, clamp(ke[r], 0, max_kv_len)) of every row r < num_rows exactly once,
 * split into `splits` contiguous segments per row (one 512-thread CTA each,
 * 256-bit loads), and writes an XOR checksum of each segment's bit patterns
 * to out[r * splits + p] (device uint32 [num_rows][splits]).  Its duration is
 * the streaming floor of a workload: the time to read the algorithmic score
 * bytes of the roofline (section 6.1's complete-row work) in a comparable
 * launch shape, with no selection work.  Enqueues one kernel on `stream`.
 * Errors: ERR_NULL_POINTER, ERR_BAD_SHAPE, ERR_BAD_PLAN (splits outside
 * [1, 1024]), ERR_MISALIGNED (4-byte alignment), ERR_CUDA. */
int exact_topk_stream_floor(const float* logits, int64_t num_rows, int64_t max_kv_len,
                            int64_t row_pitch, const int32_t* ke, uint32_t* out, int splits,
                            struct CUstream_st* stream);

/* Static description of a status code; never NULL. */
const char* exact_topk_error_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int exact_topk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_TOPK_H_ */
