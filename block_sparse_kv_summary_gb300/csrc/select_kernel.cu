// Normalised scores and block selection (CompKV, section "무엇과 다른가").
//
// One 1024-thread CTA per (sequence, KV head):
//   1. LSE_g = logsumexp over blocks of a_{g,b}, combined from the scoring
//      pass's per-item (max, sum) pairs;
//   2. S_b = sum_g u_{g,b} exp(m_a(item of b) - LSE_g)  (= sum_g phat sigma2),
//      kept in shared memory as uint32 bit patterns: S_b >= 0, so the
//      unsigned order of the bits is the numeric order;
//   3. F = {0, N-2, N-1} is always selected; the other K - 3 slots go to the
//      largest keys among blocks 1..N-3, found by an MSB-first radix select
//      (4 passes of 8-bit digits over a shared histogram); keys equal to the
//      threshold are taken in increasing block index;
//   4. the selected indices are written ascending (block-wide prefix sums).
// With N <= K every block is selected.
#include "compkv_launch.h"

namespace compkv {

constexpr int kSelThreads = 1024;

size_t select_smem_bytes(int max_cap_blocks, int G) {
  const int nch = (max_cap_blocks + kChunk - 1) / kChunk;
  return (size_t)((max_cap_blocks + 3) & ~3) * 4 + (size_t)nch * G * 4 + 64;
}

// Exclusive prefix sum of one value per thread across the CTA; returns the
// exclusive prefix and writes the total to *total.  All threads must call.
__device__ __forceinline__ int block_exclusive_scan(int x, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_buf[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v = lane < nw ? warp_buf[lane] : 0;
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += y;
    }
    if (lane < nw) warp_buf[lane] = vi - v;  // exclusive warp offsets
    if (lane == 31) warp_buf[32] = vi;
  }
  __syncthreads();
  const int res = warp_buf[warp] + incl - x;
  *total = warp_buf[32];
  __syncthreads();
  return res;
}

template <int G>
__global__ void __launch_bounds__(kSelThreads) select_kernel(LayerArgs a) {
  extern __shared__ __align__(16) uint32_t keys[];
  __shared__ float lse[kMaxG];
  __shared__ uint32_t hist[256];
  __shared__ int scan_buf[33];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_k;

  const int s = blockIdx.x / a.Hkv, h = blockIdx.x % a.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = seq_tokens(a, s);
  const int N = ceil_blocks(L);
  const int K = a.K;
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = a.chunk0[s] + h * a.nchunk[s];
  float* fch = reinterpret_cast<float*>(keys + ((N + 3) & ~3));  // [nch][G]
  int* sel_out = a.sel + ((int64_t)s * a.Hkv + h) * K;
  const int rs = rec_stride(a);

  // 1. logsumexp per query head from the per-item (max, sum) pairs
  if (warp < G) {
    const int g = warp;
    float m = -INFINITY;
    for (int c = lane; c < nch; c += 32) m = fmaxf(m, __ldcg(a.chunk_rec + (int64_t)(rec0 + c) * rs + g * (4 + a.d)));
    m = warp_max(m);
    float t = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const float* rg = a.chunk_rec + (int64_t)(rec0 + c) * rs + g * (4 + a.d);
      t += __ldcg(rg + 1) * expf(__ldcg(rg) - m);
    }
    t = warp_sum(t);
    if (lane == 0) lse[g] = m + logf(t);
  }
  __syncthreads();
  // 2. per-item factors exp(m_a - LSE_g), then S_b
  for (int i = tid; i < nch * G; i += kSelThreads) {
    const int c = i / G, g = i % G;
    fch[i] = expf(__ldcg(a.chunk_rec + (int64_t)(rec0 + c) * rs + g * (4 + a.d)) - lse[g]);
  }
  __syncthreads();
  float* scores = a.scores ? a.scores + ((int64_t)s * a.Hkv + h) * a.score_stride : nullptr;
  for (int b = tid; b < N; b += kSelThreads) {
    const int c = b / kChunk, o = b % kChunk;
    float S = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) S = fmaf(__ldcg(a.chunk_u + ((int64_t)(rec0 + c) * G + g) * kChunk + o), fch[c * G + g], S);
    S = fmaxf(S, 0.f);  // S >= 0 by construction; also maps -0 to +0
    keys[b] = __float_as_uint(S);
    if (scores) scores[b] = S;
  }
  __syncthreads();

  if (N <= K) {
    for (int i = tid; i < K; i += kSelThreads) sel_out[i] = i < N ? i : -1;
    return;
  }

  // 3. radix select of the (K-3)-th largest key among candidates 1..N-3
  uint32_t prefix = 0xffffffffu, mask = 0;
  int kk = K - 3;
  if (kk > 0) prefix = 0;  // with K = 3 only the forced blocks are taken (no key exceeds 0xffffffff)
  for (int pass = 0; pass < 4 && kk > 0; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int b = 1 + tid; b <= N - 3; b += kSelThreads) {
      const uint32_t key = keys[b];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255-8l .. 248-8l (descending); find the digit where
      // the count of larger-or-equal keys first reaches kk
      uint32_t cnt[8];
      uint32_t loc = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = hist[255 - 8 * lane - i];
        loc += cnt[i];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t before = incl - loc;
      if (before < (uint32_t)kk && (uint32_t)kk <= incl) {
        uint32_t run = before;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (run < (uint32_t)kk && (uint32_t)kk <= run + cnt[i]) {
            sh_prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
            sh_k = kk - (int)run;
          }
          run += cnt[i];
        }
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    kk = sh_k;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // key of the (K-3)-th largest candidate
  const int need_eq = kk;     // candidates equal to T to take, lowest index first

  // 4. rank ties by index, then compact ascending; thread t owns a contiguous range
  const int per = (N + kSelThreads - 1) / kSelThreads;
  const int lo = min(N, tid * per), hi = min(N, lo + per);
  int eq_cnt = 0;
  for (int b = lo; b < hi; ++b)
    if (b >= 1 && b <= N - 3 && keys[b] == T) ++eq_cnt;
  int total;
  const int eq_start = block_exclusive_scan(eq_cnt, scan_buf, &total);
  int my_sel = 0;
  {
    int rk = eq_start;
    for (int b = lo; b < hi; ++b) {
      const bool cand = b >= 1 && b <= N - 3;
      const uint32_t key = keys[b];
      my_sel += !cand || key > T || (key == T && rk++ < need_eq);
    }
  }
  int pos = block_exclusive_scan(my_sel, scan_buf, &total);
  if (tid == 0 && total != K) set_error(a.status, kDevInternal, s, h, 20);
  {
    int rk = eq_start;
    for (int b = lo; b < hi; ++b) {
      const bool cand = b >= 1 && b <= N - 3;
      const uint32_t key = keys[b];
      const bool take = !cand || key > T || (key == T && rk++ < need_eq);
      if (take && pos < K) sel_out[pos++] = b;
    }
  }
}

cudaError_t launch_select(const LayerArgs& a, int max_cap_blocks, cudaStream_t st) {
  const size_t sm = select_smem_bytes(max_cap_blocks, a.G);
  cudaError_t e = cudaSuccess;
#define COMPKV_SEL(GG)                                                                                     \
  case GG:                                                                                                 \
    e = cudaFuncSetAttribute(select_kernel<GG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);    \
    if (e != cudaSuccess) return e;                                                                        \
    select_kernel<GG><<<a.B * a.Hkv, kSelThreads, sm, st>>>(a);                                            \
    break;
  switch (a.G) {
    COMPKV_SEL(1)
    COMPKV_SEL(2)
    COMPKV_SEL(4)
    COMPKV_SEL(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef COMPKV_SEL
  return cudaGetLastError();
}

}  // namespace compkv
