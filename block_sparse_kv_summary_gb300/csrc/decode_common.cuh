// Pieces shared by the two decode kernels: the work plan both derive from the
// sequence lengths, and the stage geometry of the summary stream.
#pragma once

#include "compkv_device.cuh"

namespace compkv {

// Blocks per stream stage: 8, or 4 when the Dbar rows are long (r >= 64) or
// the group has 8 query heads (one (block, head) value per lane either way).
__host__ __device__ constexpr int stage_blocks(int r, int G) { return (r >= 64 || G >= 8) ? 4 : 8; }
// sigma2 by a butterfly over the r groups (long Dbar rows) instead of per value.
__host__ __device__ constexpr bool long_dbar(int r) { return r >= 64; }

// Blocks of sequence s the summary stream reads in this call: all of them,
// except that a call which appends leaves the open block (the one receiving
// the new token) to the post kernel, which recomputes its summary; and none
// when the call selects and every block fits the budget (K >= N) without
// scores requested: the selection is then every block and nothing of the
// summaries is needed.
__device__ __forceinline__ int streamed_blocks(int L, bool appended, bool selects, int K, bool scores) {
  const int N = ceil_blocks(L);
  if (selects && N <= K && !scores) return 0;
  return N - (appended ? 1 : 0);
}

// Per-sequence plan in shared memory, built by warp 0 from the streamed block
// counts sN[s] (s < B <= 64): soff[s] = first segment of (s, head 0),
// soff[B] = all segments, *sseg = blocks per segment.  Sequence s has
// nseg_s = ceil(sN[s] / seg) segments per head.  The caller synchronises the
// CTA afterwards.
__device__ __forceinline__ void plan_warp(const int* sN, int B, int Hkv, int P, int sb, int* soff, int* sseg, int lane) {
  const int n0 = lane < B ? sN[lane] : 0;
  const int n1 = lane + 32 < B ? sN[lane + 32] : 0;
  long long tot = (long long)n0 + n1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const int seg = plan_seg(tot * Hkv, P, sb);
  const int c0 = Hkv * ((n0 + seg - 1) / seg), c1 = Hkv * ((n1 + seg - 1) / seg);
  // exclusive prefix over sequences 0..63 (lane holds s = lane and s = lane + 32)
  int i0 = c0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, i0, o);
    if (lane >= o) i0 += y;
  }
  const int tot0 = __shfl_sync(0xffffffffu, i0, 31);
  int i1 = c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, i1, o);
    if (lane >= o) i1 += y;
  }
  if (lane < B) soff[lane] = i0 - c0;
  if (lane + 32 < B) soff[lane + 32] = tot0 + i1 - c1;
  if (lane == 0) *sseg = seg;
  if (lane == 31) soff[B] = tot0 + (B > 32 ? i1 : 0);
}

// Segment `i` of the plan: sequence, head, and its block range [b0, b0 + nb).
__device__ __forceinline__ void plan_segment(int i, int B, int Hkv, const int* sN, const int* soff, int seg, int* s,
                                             int* h, int* b0, int* nb) {
  int x = 0;
  while (x + 1 < B && soff[x + 1] <= i) ++x;
  const int per = (sN[x] + seg - 1) / seg;
  const int loc = i - soff[x];
  *s = x;
  *h = loc / per;
  const int j = loc % per;
  *b0 = j * seg;
  *nb = min(seg, sN[x] - j * seg);
}

}  // namespace compkv
