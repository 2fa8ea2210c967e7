// Host side of the exact Top-K library: the shape-stable planner ("Sample-Guided
// Exact Top-K Selection for Long-Context Sparse Attention", section 5.5,
// "Shape-stable dispatch"), workspace contract and the C ABI declared in
// include/exact_topk.h.  Nothing here synchronizes, allocates or reads device
// memory, so every entry point can run before or inside a CUDA graph capture
// (after the first call on a device has cached its attributes).

#include <cuda_runtime_api.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "etk_internal.h"

namespace etk {

namespace {

constexpr uint64_t kAlign = 256;

uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-device cache of exact_topk_device_info (the attribute queries and the
// kernel attribute setup run once per device, before any capture).
constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices];
exact_topk_device_info g_info[kMaxDevices];

int cached_device_info(exact_topk_device_info* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXACT_TOPK_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return exact_topk_query_device(dev, info);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_have[dev]) {
    const int rc = exact_topk_query_device(dev, &g_info[dev]);
    if (rc != EXACT_TOPK_OK) return rc;
    g_have[dev] = true;
  }
  *info = g_info[dev];
  return EXACT_TOPK_OK;
}

}  // namespace

WorkspaceLayout workspace_layout(const exact_topk_plan& plan) {
  WorkspaceLayout lay{};
  const int64_t N = plan.max_kv_len;
  int64_t slices = 0;
  switch (plan.family) {
    case EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED:
    case EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT:
      // One frontier slice per worker CTA, reused across the rows it claims
      // (section 5.4); needed only when a frontier can exceed shared memory.
      slices = N > plan.cand_capacity ? plan.workers : 0;
      break;
    case EXACT_TOPK_FAMILY_KV_SPLIT:
      // One row buffer per captured row: disjoint segment-owned candidate
      // ranges, then the finisher's frontier spill (section 5.5).
      slices = plan.num_rows;
      break;
    default:
      break;
  }
  uint64_t off = 0;
  lay.slices = slices;
  lay.pair_offset = off;
  off = round_up(off + (uint64_t)slices * (uint64_t)N * 8u, kAlign);
  lay.seg_offset = off;
  if (plan.family == EXACT_TOPK_FAMILY_KV_SPLIT)
    off = round_up(off + (uint64_t)plan.num_rows * (uint64_t)plan.splits * 8u, kAlign);
  lay.defer_offset = off;
  if (plan.family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED)
    off = round_up(off + (uint64_t)plan.num_rows * 32u, kAlign);
  lay.total = off;
  return lay;
}

}  // namespace etk

using namespace etk;

extern "C" {

int exact_topk_version(void) { return 10000; }

const char* exact_topk_error_string(int status) {
  switch (status) {
    case EXACT_TOPK_OK:
      return "success";
    case EXACT_TOPK_ERR_NULL_POINTER:
      return "a required pointer is NULL";
    case EXACT_TOPK_ERR_BAD_SHAPE:
      return "bad shape: need num_rows >= 1, 1 <= max_kv_len <= row_pitch <= 2^31-16";
    case EXACT_TOPK_ERR_BAD_K:
      return "bad top_k: need 1 <= top_k <= EXACT_TOPK_MAX_K";
    case EXACT_TOPK_ERR_COUNTERS_TOO_SMALL:
      return "counter buffer smaller than counter_bytes";
    case EXACT_TOPK_ERR_WORKSPACE_TOO_SMALL:
      return "workspace smaller than workspace_bytes";
    case EXACT_TOPK_ERR_MISALIGNED:
      return "misaligned buffer: scores/ke/out need 4-byte, counters/workspace 16-byte alignment";
    case EXACT_TOPK_ERR_BAD_PLAN:
      return "plan field out of range or inconsistent";
    case EXACT_TOPK_ERR_CUDA:
      return "CUDA runtime call failed";
    default:
      return "unknown exact_topk status";
  }
}

int exact_topk_query_device(int device, exact_topk_device_info* info) {
  if (info == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return EXACT_TOPK_ERR_CUDA;
  exact_topk_device_info d{};
  d.sm_count = sms;
  int rc = kernel_occupancy(EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED, device, &d.persistent_ctas_per_sm);
  if (rc != EXACT_TOPK_OK) return rc;
  rc = kernel_occupancy(EXACT_TOPK_FAMILY_KV_SPLIT, device, &d.kvsplit_ctas_per_sm);
  if (rc != EXACT_TOPK_OK) return rc;
  rc = kernel_occupancy(EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT, device, &d.rowlocal_ctas_per_sm);
  if (rc != EXACT_TOPK_OK) return rc;
  rc = kernel_occupancy(EXACT_TOPK_FAMILY_CLUSTER_SPLIT, device, &d.cluster_ctas_per_sm);
  if (rc != EXACT_TOPK_OK) return rc;
  *info = d;
  return EXACT_TOPK_OK;
}

int exact_topk_make_plan(int64_t num_rows, int64_t max_kv_len, int64_t row_pitch, int top_k,
                         const exact_topk_device_info* info, const exact_topk_plan_request* req,
                         exact_topk_plan* plan) {
  if (info == nullptr || plan == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  if (num_rows < 1 || num_rows > 0x7FFFFFFFLL || max_kv_len < 1 || max_kv_len > EXACT_TOPK_MAX_N ||
      row_pitch < max_kv_len || row_pitch > ((int64_t)1 << 40))
    return EXACT_TOPK_ERR_BAD_SHAPE;
  if (top_k < 1 || top_k > EXACT_TOPK_MAX_K) return EXACT_TOPK_ERR_BAD_K;
  if (info->sm_count < 1) return EXACT_TOPK_ERR_BAD_PLAN;
  exact_topk_plan_request r{};
  r.dual = -1;
  if (req != nullptr) r = *req;

  exact_topk_plan p{};
  p.num_rows = num_rows;
  p.max_kv_len = max_kv_len;
  p.row_pitch = row_pitch;
  p.top_k = top_k;
  p.sm_count = info->sm_count;

  // Family (section 5.5, Fig. 6).
  // - Rows narrower than 16K: row-local exact below the sampling crossover
  //   (section 6.4 places it between 16-24K and 64K columns on H20).  On
  //   GB300 the sampled path wins from 1K columns (K from 64 to 2048) once
  //   the rows need more than one wave of row-local CTAs, so the exact kernel
  //   keeps only single-wave batches and rows under 1K columns (not measured).
  // - Fewer rows than SMs: the cluster split if a row fits the shared memory
  //   of one cluster (and its CTAs fit in about two waves), else the KV-split,
  //   unless the KV-split would give each row a single segment: the
  //   persistent kernel then runs the same one-CTA-per-row work faster.
  // - Persistent sampled otherwise.
  // Cluster split: the fewest CTAs that hold the row in shared memory, up to
  // 16; rows up to 16 * kClusterSegment scores leave the rest of each
  // segment in global memory.
  const int64_t cluster_min_P = ceil_div64(max_kv_len, kClusterSegment);
  const int64_t held_P = ceil_div64(max_kv_len, kClusterStage);
  const int64_t cluster_P = held_P < kClusterMaxSplits ? held_P : kClusterMaxSplits;
  const bool cluster_fits = cluster_min_P <= kClusterMaxSplits;
  const int64_t rowlocal_wave =
      (int64_t)info->sm_count * (info->rowlocal_ctas_per_sm > 0 ? info->rowlocal_ctas_per_sm : 1);
  const int64_t kv_target =
      (int64_t)info->sm_count * (info->kvsplit_ctas_per_sm > 0 ? info->kvsplit_ctas_per_sm : 1) / 4;
  int family = r.family;
  if (family == EXACT_TOPK_FAMILY_AUTO) {
    if (max_kv_len < 16384)
      family = (max_kv_len >= 1024 && num_rows > rowlocal_wave)
                   ? EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED
                   : EXACT_TOPK_FAMILY_ROW_LOCAL_EXACT;
    else if (num_rows < info->sm_count)
      // The planner takes clusters of up to 8 CTAs (rows up to 131072 scores,
      // held in shared memory).  Clusters of up to 16, whose segments read
      // their second half from global memory, run on request: on the few
      // long rows workload (8 x 524288) they measured 35.4 us against 30.9 us
      // for the KV-split.
      family = (cluster_fits && cluster_P <= 8 && info->cluster_ctas_per_sm > 0 &&
                num_rows * cluster_P <= 2LL * info->sm_count * info->cluster_ctas_per_sm)
                   ? EXACT_TOPK_FAMILY_CLUSTER_SPLIT
                   : (num_rows >= kv_target ? EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED
                                            : EXACT_TOPK_FAMILY_KV_SPLIT);
    else
      family = EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED;
  }
  if (family < EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED || family > EXACT_TOPK_FAMILY_CLUSTER_SPLIT)
    return EXACT_TOPK_ERR_BAD_PLAN;
  p.family = family;

  // View density and boundary policy (section 5.5: stride-64 and stride-128
  // policies; the wide-row policy keeps the secondary boundary).
  const int64_t stride = r.stride ? r.stride : (max_kv_len < 65536 ? 64 : 128);
  if (!is_pow2(stride) || stride < 2 || stride > 4096) return EXACT_TOPK_ERR_BAD_PLAN;
  p.stride = (int32_t)stride;
  if (r.dual < -1 || r.dual > 1) return EXACT_TOPK_ERR_BAD_PLAN;
  p.dual = r.dual >= 0 ? r.dual : (max_kv_len >= 65536 ? 1 : 0);
  // Retention margins: K~ = 1.5K (section 4.2) and K~1 = 1.75K (section 6.4).
  p.rho0_num = r.rho0_num ? r.rho0_num : 3;
  p.rho0_den = r.rho0_den ? r.rho0_den : 2;
  p.rho1_num = r.rho1_num ? r.rho1_num : 7;
  p.rho1_den = r.rho1_den ? r.rho1_den : 4;
  if (p.rho0_num < 1 || p.rho0_den < 1 || p.rho1_num < 1 || p.rho1_den < 1 ||
      p.rho0_num > 1024 || p.rho0_den > 1024 || p.rho1_num > 1024 || p.rho1_den > 1024)
    return EXACT_TOPK_ERR_BAD_PLAN;
  // q = ceil(K~ / s)  (eq. 15)
  p.q0 = (int32_t)ceil_div64((int64_t)p.rho0_num * top_k, (int64_t)p.rho0_den * stride);
  p.q1 = (int32_t)ceil_div64((int64_t)p.rho1_num * top_k, (int64_t)p.rho1_den * stride);
  if (p.dual && p.q1 < p.q0) return EXACT_TOPK_ERR_BAD_PLAN;

  int ctas_per_sm = 1;
  switch (family) {
    case EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED:
      p.threads = kPersistentThreads;
      p.cand_capacity = kPersistentCap;
      ctas_per_sm = info->persistent_ctas_per_sm;
      break;
    case EXACT_TOPK_FAMILY_KV_SPLIT:
      p.threads = kKvSplitThreads;
      p.cand_capacity = kKvSplitCap;
      ctas_per_sm = info->kvsplit_ctas_per_sm;
      break;
    case EXACT_TOPK_FAMILY_CLUSTER_SPLIT:
      p.threads = kClusterThreads;
      p.cand_capacity = kClusterStage;
      ctas_per_sm = info->cluster_ctas_per_sm;
      break;
    default:
      p.threads = kRowLocalThreads;
      p.cand_capacity = kRowLocalCap;
      ctas_per_sm = info->rowlocal_ctas_per_sm;
      break;
  }
  if (ctas_per_sm < 1) ctas_per_sm = 1;

  if (family == EXACT_TOPK_FAMILY_KV_SPLIT) {
    // P: enough segment CTAs to cover about a quarter of the device's resident
    // CTA slots, with segments of at least 8K scores (section 4.6: KV-split
    // trades replicated view work, R_eq = 1 + P/s, for a shorter validation
    // span; on GB300 the few-long-rows workload is fastest at this P).
    int64_t P = r.splits;
    if (P == 0) {
      const int64_t target = kv_target;
      P = 1;
      while (P < 64 && num_rows * P < target) P *= 2;
      while (P > 1 && max_kv_len / P < 8192) P /= 2;
    }
    if (P < 1 || P > 128 || num_rows > 65535) return EXACT_TOPK_ERR_BAD_PLAN;
    p.splits = (int32_t)P;
    p.workers = (int32_t)(num_rows * P);
  } else if (family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT) {
    const int64_t P = r.splits ? r.splits : cluster_P;
    if (P < cluster_min_P || P > kClusterMaxSplits || num_rows > 65535)
      return EXACT_TOPK_ERR_BAD_PLAN;
    p.splits = (int32_t)P;
    p.workers = (int32_t)(num_rows * P);
  } else {
    int64_t W = r.workers ? r.workers : (int64_t)info->sm_count * ctas_per_sm;
    if (W < 1) return EXACT_TOPK_ERR_BAD_PLAN;
    if (W > num_rows) W = num_rows;
    p.workers = (int32_t)W;
    p.splits = 1;
  }

  p.counter_bytes = round_up((uint64_t)(kCtrArriveBase + num_rows) * 4u, 16);
  p.workspace_bytes = workspace_layout(p).total;
  *plan = p;
  return EXACT_TOPK_OK;
}

int exact_topk_workspace_size(int64_t num_rows, int64_t max_kv_len, int top_k,
                              size_t* counter_bytes, size_t* workspace_bytes) {
  if (counter_bytes == nullptr || workspace_bytes == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  exact_topk_device_info info;
  int rc = cached_device_info(&info);
  if (rc != EXACT_TOPK_OK) return rc;
  exact_topk_plan plan;
  rc = exact_topk_make_plan(num_rows, max_kv_len, max_kv_len, top_k, &info, nullptr, &plan);
  if (rc != EXACT_TOPK_OK) return rc;
  *counter_bytes = (size_t)plan.counter_bytes;
  *workspace_bytes = (size_t)plan.workspace_bytes;
  return EXACT_TOPK_OK;
}

}  // extern "C"

namespace etk {

int check_run(const exact_topk_plan* plan, const float* logits, const int32_t* ke,
              const int32_t* out, const int32_t* num_valid_rows, const void* counters,
              size_t counter_bytes, const void* workspace, size_t workspace_bytes,
              const int32_t* prev_topk, const int32_t* trace) {
  if (plan == nullptr || logits == nullptr || ke == nullptr || out == nullptr ||
      counters == nullptr)
    return EXACT_TOPK_ERR_NULL_POINTER;
  if (plan->workspace_bytes > 0 && workspace == nullptr) return EXACT_TOPK_ERR_NULL_POINTER;
  if (plan->num_rows < 1 || plan->max_kv_len < 1 || plan->max_kv_len > EXACT_TOPK_MAX_N ||
      plan->row_pitch < plan->max_kv_len)
    return EXACT_TOPK_ERR_BAD_SHAPE;
  if (plan->top_k < 1 || plan->top_k > EXACT_TOPK_MAX_K) return EXACT_TOPK_ERR_BAD_K;
  if (plan->family < EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED ||
      plan->family > EXACT_TOPK_FAMILY_CLUSTER_SPLIT || plan->workers < 1 ||
      plan->splits < 1 || plan->stride < 2 || !is_pow2(plan->stride) || plan->q0 < 1 ||
      plan->q1 < 1 || (plan->dual != 0 && plan->dual != 1))
    return EXACT_TOPK_ERR_BAD_PLAN;
  if (plan->family == EXACT_TOPK_FAMILY_KV_SPLIT &&
      (plan->num_rows > 65535 || plan->splits > 128 ||
       (int64_t)plan->workers != plan->num_rows * plan->splits))
    return EXACT_TOPK_ERR_BAD_PLAN;
  if (plan->family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT &&
      (plan->num_rows > 65535 || plan->splits > kClusterMaxSplits ||
       (int64_t)plan->splits * kClusterSegment < plan->max_kv_len ||
       (int64_t)plan->workers != plan->num_rows * plan->splits))
    return EXACT_TOPK_ERR_BAD_PLAN;
  const int expect_cap = plan->family == EXACT_TOPK_FAMILY_PERSISTENT_SAMPLED
                             ? kPersistentCap
                             : (plan->family == EXACT_TOPK_FAMILY_KV_SPLIT
                                    ? kKvSplitCap
                                    : (plan->family == EXACT_TOPK_FAMILY_CLUSTER_SPLIT
                                           ? kClusterStage
                                           : kRowLocalCap));
  if (plan->cand_capacity != expect_cap) return EXACT_TOPK_ERR_BAD_PLAN;
  const WorkspaceLayout lay = workspace_layout(*plan);
  if (lay.total != plan->workspace_bytes) return EXACT_TOPK_ERR_BAD_PLAN;
  if (counter_bytes < plan->counter_bytes) return EXACT_TOPK_ERR_COUNTERS_TOO_SMALL;
  if (workspace_bytes < plan->workspace_bytes) return EXACT_TOPK_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(logits, 4) || !aligned(ke, 4) || !aligned(out, 4) || !aligned(counters, 16) ||
      (workspace != nullptr && !aligned(workspace, 16)) ||
      (num_valid_rows != nullptr && !aligned(num_valid_rows, 4)) ||
      (prev_topk != nullptr && !aligned(prev_topk, 4)) || (trace != nullptr && !aligned(trace, 4)))
    return EXACT_TOPK_ERR_MISALIGNED;
  return EXACT_TOPK_OK;
}

}  // namespace etk

extern "C" {

int exact_topk_run(const exact_topk_plan* plan, const float* logits, const int32_t* ke,
                   int32_t* out, const int32_t* num_valid_rows, void* counters,
                   size_t counter_bytes, void* workspace, size_t workspace_bytes,
                   const int32_t* prev_topk, int32_t* trace, struct CUstream_st* stream) {
  const int rc = check_run(plan, logits, ke, out, num_valid_rows, counters, counter_bytes,
                           workspace, workspace_bytes, prev_topk, trace);
  if (rc != EXACT_TOPK_OK) return rc;
  LaunchArgs a;
  a.logits = logits;
  a.ke = ke;
  a.out = out;
  a.num_valid_rows = num_valid_rows;
  a.counters = counters;
  a.workspace = workspace;
  a.prev_topk = prev_topk;
  a.trace = trace;
  return launch(*plan, a, reinterpret_cast<cudaStream_t>(stream));
}

int exact_topk(const float* logits, int64_t num_rows, int64_t max_kv_len, const int32_t* ke,
               int32_t* out, const int32_t* num_valid_rows, int top_k, void* counters,
               size_t counter_bytes, void* workspace, size_t workspace_bytes,
               const int32_t* prev_topk, struct CUstream_st* stream) {
  if (logits == nullptr || ke == nullptr || out == nullptr || counters == nullptr)
    return EXACT_TOPK_ERR_NULL_POINTER;
  exact_topk_device_info info;
  int rc = cached_device_info(&info);
  if (rc != EXACT_TOPK_OK) return rc;
  exact_topk_plan plan;
  rc = exact_topk_make_plan(num_rows, max_kv_len, max_kv_len, top_k, &info, nullptr, &plan);
  if (rc != EXACT_TOPK_OK) return rc;
  return exact_topk_run(&plan, logits, ke, out, num_valid_rows, counters, counter_bytes, workspace,
                        workspace_bytes, prev_topk, nullptr, stream);
}

}  // extern "C"
