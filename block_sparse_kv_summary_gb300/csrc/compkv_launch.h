// Host-side launchers of the CompKV kernels, shared between the kernel
// translation units and the C-ABI dispatch.
#pragma once

#include <cuda_runtime.h>

#include "compkv_device.cuh"

namespace compkv {

// Parts of the decode step a call runs.
enum FusedFlags : int {
  kFAppend = 1,   // pack the new token and recompute the open block's summary
  kFScore = 2,    // sigma2, a = ln|b| + zbar + sigma2/2 and its logsumexp parts
  kFComp = 4,     // zbar per block and the compensation sums
  kFSelect = 8,   // LSE, S_b, forced set + Top-K
  kFAttend = 16,  // exact attention over the selection + Mean compensation
};
constexpr int kFusedDecode = kFAppend | kFScore | kFComp | kFSelect | kFAttend;
constexpr int kFusedScoreSelect = kFScore | kFSelect;
constexpr int kFusedAttend = kFComp | kFAttend;
constexpr int kMaxStreamCtas = 1024;   // the stream kernel's grid at most (segment records: this + units)

cudaError_t launch_prefill(const LayerArgs& a, int64_t rows_per_layer, cudaStream_t st);
cudaError_t launch_append(const LayerArgs& a, cudaStream_t st);
// Copies three buffers (byte counts multiples of 16, 16-byte aligned) to device memory in one
// kernel; the sources may be page-locked host memory.
cudaError_t launch_stage_in(void* d0, const void* s0, size_t b0, void* d1, const void* s1, size_t b1, void* d2,
                            const void* s2, size_t b2, cudaStream_t st);
// One bounded mbarrier wait that runs out and records kDevTimeout in `status`.
cudaError_t launch_wait_selftest(int* status, cudaStream_t st);

// The decode step is two kernels on `st`, chained by programmatic dependent
// launch: the summary stream over every block (a.P persistent CTAs), then one
// cluster of a.C CTAs per (sequence, KV head) for the selection, attention
// and compensation.  `mode` is kFusedDecode, kFusedScoreSelect or
// kFusedAttend.
// A call that appends gives the first Q CTAs of the stream kernel's grid the
// open blocks (one warp per unit, at most 8 CTAs) and leaves P - Q CTAs to the
// summary stream; both launches of a chain apply the same split.
inline void chain_split(LayerArgs& a, int mode) {
  a.Q = 0;
  if (mode & kFAppend) {
    int q = (a.B * a.Hkv + 7) / 8;
    if (q > 8) q = 8;
    a.Q = q;
    a.P = a.P > q ? a.P - q : 1;
  }
}
cudaError_t launch_stream(const LayerArgs& a, int mode, cudaStream_t st, bool pdl);
cudaError_t launch_post(const LayerArgs& a, int mode, cudaStream_t st);

// Function attributes the launches need, set once per context (compkv_init) instead of on
// every launch: the dynamic shared memory limit of every mode's stream and post kernel raised
// (never lowered: another context may need more) to this configuration's, and clusters of
// more than 8 CTAs allowed.
inline cudaError_t raise_smem_limit(const void* fn, int smem) {
  cudaFuncAttributes at;
  cudaError_t e = cudaFuncGetAttributes(&at, fn);
  if (e != cudaSuccess) return e;
  if (at.maxDynamicSharedSizeBytes >= smem) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}
cudaError_t prepare_stream(int D, int r, int G);
cudaError_t prepare_post(int D, int G, int C, int bpc_max, int K);

// Dynamic shared memory of the two kernels.
size_t stream_smem(int D, int r, int G);
size_t post_smem(int D, int G, int C, int bpc_max, int K);
// Stream CTAs resident per multiprocessor (occupancy of the decode variant).
int stream_ctas_per_sm(int D, int r, int G);

}  // namespace compkv
