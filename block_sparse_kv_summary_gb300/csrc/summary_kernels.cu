// Block summaries {|b|, kbar_b, Dbar_b, vbar_b} (CompKV, section "무엇과 다른가"):
// the bulk build over a prefilled cache, and the per-step append that packs the
// new token and recomputes the open block ("어떻게 쓰나": the fused kernel that
// updates the current block's statistics and packs the new K/V).
//
// One warp summarises one block: lane l holds D/32 consecutive coordinates of
// every token.  Mean and population variance are two-pass in fp32 from the
// exact bf16 values (one pass over registers for the mean, one for the
// squared deviations), so no E[k^2] - E[k]^2 cancellation.
#include "compkv_launch.h"

namespace compkv {

template <int D>
__device__ __forceinline__ void warp_block_summary(const __nv_bfloat16* krow, const __nv_bfloat16* vrow, int n,
                                                   const __nv_bfloat16* knew, const __nv_bfloat16* vnew,
                                                   float* kbar, float* vbar, float* dbar, int r, int lane) {
  constexpr int V = D / 32;
  float kt[kBlock][V];
  float ks[V], vs[V];
#pragma unroll
  for (int i = 0; i < V; ++i) ks[i] = vs[i] = 0.f;
#pragma unroll
  for (int j = 0; j < kBlock; ++j) {
    if (j < n) {
      const bool is_new = (knew != nullptr) && (j == n - 1);
      const __nv_bfloat16* kp = is_new ? knew + lane * V : krow + j * D + lane * V;
      const __nv_bfloat16* vp = is_new ? vnew + lane * V : vrow + j * D + lane * V;
      float vf[V];
      load_bf16<V>(kp, kt[j]);
      load_bf16<V>(vp, vf);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        ks[i] += kt[j][i];
        vs[i] += vf[i];
      }
    }
  }
  const float fn = (float)n;
  float mean[V], var[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    mean[i] = ks[i] / fn;
    var[i] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < kBlock; ++j) {
    if (j < n) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float dlt = kt[j][i] - mean[i];
        var[i] = fmaf(dlt, dlt, var[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    var[i] = var[i] / fn;
    kbar[lane * V + i] = mean[i];
    vbar[lane * V + i] = vs[i] / fn;
  }
  // grouped mean of the variances: group t = coordinates [t*D/r, (t+1)*D/r)
  const int gs = D / r;
  if (gs >= V) {
    const int lpg = gs / V;  // lanes per group (power of two)
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) t += var[i];
    for (int o = lpg >> 1; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((lane & (lpg - 1)) == 0) dbar[lane / lpg] = t / (float)gs;
  } else {
    const int per = V / gs;  // groups per lane
    for (int t = 0; t < per; ++t) {
      float sum = 0.f;
      for (int c = 0; c < gs; ++c) sum += var[t * gs + c];
      dbar[lane * per + t] = sum / (float)gs;
    }
  }
}

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
  const int L = a.seq_len[s];
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

cudaError_t launch_append(const LayerArgs& a, cudaStream_t st) {
  const int threads = 32 * a.Hkv;
  if (a.d == 128)
    append_kernel<128><<<a.B, threads, 0, st>>>(a);
  else
    append_kernel<64><<<a.B, threads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace compkv
