// Internal interface between the host planner / C ABI (exact_topk_api.cpp)
// and the kernel translation unit (topk_kernels.cu).  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime_api.h>

#include "exact_topk.h"

namespace etk {

// Counter buffer layout (int32 words).  The queue head and exit counter drive
// the persistent row queue; arrive[r] elects the KV-split finisher of row r;
// status is a sticky error word that stays zero unless a device-side bounds
// guard tripped; the deferred count hands rows from the persistent kernel to
// the heavy-row kernel that follows it.  Every call returns words 0, 1, 3 and
// arrive[] to zero.
constexpr int kCtrQueue = 0;
constexpr int kCtrExit = 1;
constexpr int kCtrStatus = 2;
constexpr int kCtrDeferred = 3;  // persistent family: rows handed to the heavy-row kernel
constexpr int kCtrArriveBase = 4;

#ifndef ETK_PERSISTENT_THREADS
#define ETK_PERSISTENT_THREADS 512
#endif
#ifndef ETK_PERSISTENT_CAP
#define ETK_PERSISTENT_CAP 5376
#endif
// Persistent sampled kernel: CTA size (1024 / kPersistentThreads CTAs per SM)
// and on-chip frontier entries.  5376 entries (42 KB) is the most that keeps
// two CTAs on an SM's 228 KB of shared memory with room to spare; on the
// causal prefill batch (K = 2048) the frontier after Phase 2 has a median of
// about 3300 entries and a 99th percentile of about 5100, and a frontier
// beyond the capacity refines from global memory without the next row's
// Phase 1 beside it (4096 entries: 14% of the rows spilled, 418 us; 5376:
// 407 us).
constexpr int kPersistentThreads = ETK_PERSISTENT_THREADS;
constexpr int kKvSplitThreads = 512;
constexpr int kRowLocalThreads = 1024;
constexpr int kClusterThreads = 512;
// Cluster split: scores of a row segment held in a CTA's shared memory, the
// longest segment of one CTA (the rest read from global memory), and the
// largest cluster (16: above the portable limit of 8, allowed per kernel).
constexpr int kClusterStage = 16384;
constexpr int kClusterSegment = 2 * kClusterStage;
constexpr int kClusterMaxSplits = 16;
constexpr int kPersistentCap = ETK_PERSISTENT_CAP;
constexpr int kKvSplitCap = 4096;
constexpr int kRowLocalCap = 8192;
// Rows of the row-local exact kernel up to this length stay in registers.
constexpr int kRowLocalResident = 8 * kRowLocalThreads;

struct LaunchArgs {
  const float* logits;
  const int32_t* ke;
  int32_t* out;
  const int32_t* num_valid_rows;
  void* counters;
  void* workspace;
  const int32_t* prev_topk;
  int32_t* trace;
};

// Bytes of dynamic shared memory a kernel of `family` uses for a frontier of
// `cap` entries.
size_t shared_bytes(int family, int cap);

// Workspace carve-up shared by the planner and the launcher.
struct WorkspaceLayout {
  uint64_t pair_offset;   // (int32 index, uint32 key) pairs [slices][N]
  uint64_t seg_offset;    // int32 pairs [M][P] (KV-split published counts)
  uint64_t defer_offset;  // persistent family: int32 [M][8] deferred-row records
  uint64_t total;
  int64_t slices;
};
WorkspaceLayout workspace_layout(const exact_topk_plan& plan);

// Every host-side check of exact_topk_run (pointers, shapes, plan
// consistency, buffer sizes, alignment); EXACT_TOPK_OK or the error status.
int check_run(const exact_topk_plan* plan, const float* logits, const int32_t* ke,
              const int32_t* out, const int32_t* num_valid_rows, const void* counters,
              size_t counter_bytes, const void* workspace, size_t workspace_bytes,
              const int32_t* prev_topk, const int32_t* trace);

// Implemented in topk_kernels.cu.
int kernel_occupancy(int family, int device, int* ctas_per_sm);
int launch(const exact_topk_plan& plan, const LaunchArgs& args, cudaStream_t stream);

}  // namespace etk
