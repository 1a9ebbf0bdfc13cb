// Host-side launchers of the CompKV kernels (one per kernel family), shared
// between the kernel translation units and the C-ABI dispatch.
#pragma once

#include <cuda_runtime.h>

#include "compkv_device.cuh"

namespace compkv {

// Parts of the decode step a fused launch runs.
enum FusedFlags : int {
  kFAppend = 1,   // pack the new token and recompute the open block's summary
  kFScore = 2,    // sigma2, a = ln|b| + zbar + sigma2/2 and the per-item logsumexp parts
  kFComp = 4,     // zbar per block and the per-item compensation sums
  kFSelect = 8,   // LSE, S_b, forced set + Top-K
  kFAttend = 16,  // exact attention over the selection + Mean compensation
};
constexpr int kFusedDecode = kFAppend | kFScore | kFComp | kFSelect | kFAttend;
constexpr int kFusedScoreSelect = kFScore | kFSelect;
constexpr int kFusedAttend = kFComp | kFAttend;
constexpr int kAttendBlocks = 12;  // selected blocks per attention work item (= consumer warps)

cudaError_t launch_prefill(const LayerArgs& a, int64_t rows_per_layer, cudaStream_t st);
cudaError_t launch_append(const LayerArgs& a, cudaStream_t st);
cudaError_t launch_fused(const LayerArgs& a, int mode, int grid, cudaStream_t st);

int fused_region_bytes(int D, int r, int G, int max_cap_blocks);
int fused_stages(int D, int r, int G, int max_cap_blocks, size_t smem_limit);
size_t fused_smem_bytes(int D, int r, int G, int max_cap_blocks, int stages);

}  // namespace compkv
