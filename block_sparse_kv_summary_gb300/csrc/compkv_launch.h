// Host-side launchers of the CompKV kernels (one per kernel family), shared
// between the kernel translation units and the C-ABI dispatch.
#pragma once

#include <cuda_runtime.h>

#include "compkv_device.cuh"

namespace compkv {

// Parts of the decode step a launch chain runs.
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
constexpr int kAttendBlocks = 8;  // selected blocks per CTA of a unit's cluster and round (one per warp)

cudaError_t launch_prefill(const LayerArgs& a, int64_t rows_per_layer, cudaStream_t st);
cudaError_t launch_append(const LayerArgs& a, cudaStream_t st);
// One bounded mbarrier wait that runs out and records kDevTimeout in `status`.
cudaError_t launch_wait_selftest(int* status, cudaStream_t st);

// The decode step as a chain of two kernels on `st` (score with the
// compensation partials; select and attend), chained with programmatic
// dependent launch.  `mode` is one of
// kFusedDecode, kFusedScoreSelect (score, select) or kFusedAttend (score for
// zbar, compensation, attend a caller-given selection).  `first_pdl` lets the
// first kernel overlap the tail of the previous work on the stream.
// `ev`: null, or four events recorded before and after each of the two kernels.
cudaError_t launch_decode_chain(const LayerArgs& a, int mode, cudaStream_t st, int first_pdl, cudaEvent_t* ev = nullptr);
// Kernels a chain of `mode` launches.
inline int chain_kernels(int mode) { return 2; }
// Largest dynamic shared memory the chain asks for.
size_t chain_smem_bytes(int D, int r, int G, int key_stride, int post_cpc, int K, int splits);

}  // namespace compkv
