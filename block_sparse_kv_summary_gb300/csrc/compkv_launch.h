// Host-side launchers of the CompKV kernels (one per kernel family), shared
// between the kernel translation units and the C-ABI dispatch.
#pragma once

#include <cuda_runtime.h>

#include "compkv_device.cuh"

namespace compkv {

// Which parts of the scoring pass to run.
enum ScoreMode : int {
  kModeScore = 1,   // z, sigma2, a = ln|b| + z + sigma2/2 and the per-chunk logsumexp parts
  kModeComp = 2,    // compensation parts: zbar per block, sum_b |b| e^{zbar} vbar_b per chunk
};

cudaError_t launch_prefill(const LayerArgs& a, int64_t rows_per_layer, cudaStream_t st);
cudaError_t launch_append(const LayerArgs& a, cudaStream_t st);
cudaError_t launch_score(const LayerArgs& a, int mode, int total_records, cudaStream_t st);
cudaError_t launch_select(const LayerArgs& a, int max_cap_blocks, cudaStream_t st);
cudaError_t launch_attend(const LayerArgs& a, cudaStream_t st);

size_t select_smem_bytes(int max_cap_blocks, int G);
size_t score_smem_bytes(int d, int r, int G, int mode);

}  // namespace compkv
