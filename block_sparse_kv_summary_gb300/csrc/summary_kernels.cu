// Block summaries {|b|, kbar_b, Dbar_b, vbar_b} (CompKV, section "무엇과 다른가"):
// the bulk build over a prefilled cache, and the per-step append that packs the
// new token and recomputes the open block ("어떻게 쓰나": the fused kernel that
// updates the current block's statistics and packs the new K/V).
//
// One warp summarises one block (block_summary.cuh).
#include "block_summary.cuh"
#include "compkv_launch.h"

namespace compkv {

// One warp per cache row of the layer; rows beyond a sequence's length are skipped.
template <int D>
__global__ void __launch_bounds__(256) prefill_kernel(LayerArgs a, int64_t rows_per_layer) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows_per_layer;
       row += warps) {
    int s = 0;
    while (s + 1 < a.B && a.seq_row0[s + 1] <= row) ++s;
    const int64_t local = row - a.seq_row0[s];
    const int b = (int)(local % a.cap_blocks[s]);
    const int L = a.lens[s];
    const int N = ceil_blocks(L);
    if (b >= N) continue;
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    warp_block_summary<D>(a.k + row * kBlock * D, a.v + row * kBlock * D, n, nullptr, nullptr, a.kbar + row * D,
                          a.vbar + row * D, a.dbar + row * a.r, a.r, lane);
  }
  if (blockIdx.x == 0 && threadIdx.x < a.B) a.seq_len[threadIdx.x] = a.lens[threadIdx.x];
}

// One CTA per sequence, one warp per KV head.  Writes token L (L = seq_len)
// into slot L % 16 of block L / 16, recomputes that block's summary from its
// L % 16 + 1 tokens and sets seq_len = L + 1.
template <int D>
__global__ void append_kernel(LayerArgs a) {
  constexpr int V = D / 32;
  const int s = blockIdx.x;
  const int h = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int L = __ldcg(a.seq_len + s);
  const bool fits = L >= 0 && L < a.cap_blocks[s] * kBlock;
  if (h < a.Hkv && fits) {
    const int b = L / kBlock, slot = L % kBlock;
    const int64_t row = row_of(a, s, h, b);
    const __nv_bfloat16* kn = a.k_new + ((int64_t)s * a.Hkv + h) * D;
    const __nv_bfloat16* vn = a.v_new + ((int64_t)s * a.Hkv + h) * D;
    store_bf16_raw<V>(a.k + (row * kBlock + slot) * D + lane * V, kn + lane * V);
    store_bf16_raw<V>(a.v + (row * kBlock + slot) * D + lane * V, vn + lane * V);
    warp_block_summary<D>(a.k + row * kBlock * D, a.v + row * kBlock * D, slot + 1, kn, vn, a.kbar + row * D,
                          a.vbar + row * D, a.dbar + row * a.r, a.r, lane);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (fits)
      a.seq_len[s] = L + 1;
    else
      set_error(a.status, kDevCapacity, s, -1, 1);
  }
}

cudaError_t launch_prefill(const LayerArgs& a, int64_t rows_per_layer, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t ctas = (rows_per_layer + 7) / 8;
  if (ctas > (int64_t)sms * 16) ctas = (int64_t)sms * 16;
  if (ctas < 1) ctas = 1;
  if (a.d == 128)
    prefill_kernel<128><<<(unsigned)ctas, 256, 0, st>>>(a, rows_per_layer);
  else
    prefill_kernel<64><<<(unsigned)ctas, 256, 0, st>>>(a, rows_per_layer);
  return cudaGetLastError();
}

// A bounded wait that runs out: one thread waits on an mbarrier whose
// transaction (16 bytes posted, never delivered) nothing completes; the wait
// gives up after its poll cap and records kDevTimeout in `status`.
__global__ void wait_selftest_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(&bar, 16u);
  mbar_wait_bounded(&bar, 0u, status, -1, -1, 90);
}

cudaError_t launch_wait_selftest(int* status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

// Copies up to three buffers of 16-byte chunks (src may be page-locked host
// memory the device reads over its link) into device memory, one chunk per
// thread and step: the inputs of a host-to-host decode call in one launch.
__global__ void stage_in_kernel(uint4* d0, const uint4* s0, int n0, uint4* d1, const uint4* s1, int n1, uint4* d2,
                                const uint4* s2, int n2) {
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n0 + n1 + n2; i += stride) {
    if (i < n0) d0[i] = __ldcg(s0 + i);
    else if (i < n0 + n1) d1[i - n0] = __ldcg(s1 + i - n0);
    else d2[i - n0 - n1] = __ldcg(s2 + i - n0 - n1);
  }
}

cudaError_t launch_stage_in(void* d0, const void* s0, size_t b0, void* d1, const void* s1, size_t b1, void* d2,
                            const void* s2, size_t b2, cudaStream_t st) {
  const int n0 = (int)(b0 / 16), n1 = (int)(b1 / 16), n2 = (int)(b2 / 16);
  const int n = n0 + n1 + n2;
  const int threads = 256, blocks = (n + threads - 1) / threads < 8 ? (n + threads - 1) / threads : 8;
  stage_in_kernel<<<blocks < 1 ? 1 : blocks, threads, 0, st>>>(
      reinterpret_cast<uint4*>(d0), reinterpret_cast<const uint4*>(s0), n0, reinterpret_cast<uint4*>(d1),
      reinterpret_cast<const uint4*>(s1), n1, reinterpret_cast<uint4*>(d2), reinterpret_cast<const uint4*>(s2), n2);
  return cudaGetLastError();
}

cudaError_t launch_append(const LayerArgs& a, cudaStream_t st) {
  const int threads = 32 * a.Hkv;
  if (a.d == 128)
    append_kernel<128><<<a.B, threads, 0, st>>>(a);
  else
    append_kernel<64><<<a.B, threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace compkv
