// Exact attention over the selected blocks plus Mean compensation for the
// others, jointly normalised (CompKV, sections "무엇과 다른가" and
// "어떻게 동작하나").
//
// Work item = up to 8 selected blocks of one (sequence, KV head); CTA of 8
// warps, warp w owns selected block w of the item.  Thread 0 gathers the
// item's K and V blocks (4 KiB each at d = 128) into shared memory with 1-D
// bulk copies.  Each warp keeps, per query head g, a running (m, l, acc) in
// the log-sum-exp form and folds into it:
//   + exp(z_j - m) and exp(z_j - m) v_j for the 16 tokens of its block,
//   - exp(ln|b| + zbar_b - m) and that times vbar_b: the block's own Mean
//     compensation term, which the scoring pass already added for every block;
//   + the scoring pass's per-item compensation sums assigned to this work item.
// So numerator and denominator are  sum_{selected tokens} + sum_{unselected
// blocks} |b| e^{zbar} (vbar, 1).  By Jensen, sum_{j in b} e^{z_j} >=
// |b| e^{zbar_b}, so each warp's denominator stays non-negative.  The warps
// are merged in shared memory, the work items of a (sequence, head) by the
// last one to finish (an arrival counter), which writes out = acc / l.
// If every block is selected the compensation terms are skipped (exact
// dense attention).
#include "compkv_launch.h"

namespace compkv {

template <int D>
struct InvSqrtDA;
template <>
struct InvSqrtDA<64> {
  static constexpr float v = 0.125f;
};
template <>
struct InvSqrtDA<128> {
  static constexpr float v = 0.08838834764831845f;
};

__device__ __forceinline__ float ln_count_a(int n) { return n == kBlock ? 2.772588722239781f : logf((float)n); }

// fold one (exponent e, weight scale) term into a running max / sum
__device__ __forceinline__ void rescale_to(float& m, float e, float& fold_old, float& fold_new) {
  const float mn = fmaxf(m, e);
  fold_old = (m == -INFINITY) ? 0.f : expf(m - mn);
  fold_new = expf(e - mn);
  m = mn;
}

template <int D, int G>
__global__ void __launch_bounds__(256) attend_kernel(LayerArgs a) {
  constexpr int V = D / 32;
  constexpr int NW = 8;
  constexpr int kBlockElems = kBlock * D;
  extern __shared__ __align__(128) __nv_bfloat16 kv_smem[];  // [NW][2][16][D]
  __shared__ float red_m[NW][G], red_l[NW][G];
  __shared__ __align__(16) float red_acc[NW][G][D];
  __shared__ int sh_nsel;
  __shared__ int sh_last;
  __shared__ __align__(8) uint64_t bar;

  const int split = blockIdx.x % a.splits;
  const int sh = blockIdx.x / a.splits;
  const int s = sh / a.Hkv, h = sh % a.Hkv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = seq_tokens(a, s);
  const int N = ceil_blocks(L);
  const int K = a.K;
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = a.chunk0[s] + h * a.nchunk[s];
  const int* selrow = a.sel + ((int64_t)s * a.Hkv + h) * K;

  // validate the selection row and count its valid entries
  if (tid == 0) sh_nsel = 0;
  __syncthreads();
  {
    int cnt = 0;
    bool bad = false;
    for (int i = tid; i < K; i += 256) {
      const int e = selrow[i];
      const int prev = i > 0 ? selrow[i - 1] : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      cnt += ok;
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    if (lane == 0 && cnt) atomicAdd(&sh_nsel, cnt);
    if (bad && split == 0) set_error(a.status, kDevBadSelection, s, h, 30);
  }
  // my block, and the gather
  const int my_i = split * kSplitBlocks + warp;
  int my_b = -1;
  if (my_i < K) {
    const int e = selrow[my_i];
    const int prev = my_i > 0 ? selrow[my_i - 1] : -1;
    if (e >= 0 && e < N && (my_i == 0 || (prev >= 0 && prev < e))) my_b = e;
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool comp = sh_nsel < N;
  if (tid == 0) {
    uint32_t total = 0;
    int bl[kSplitBlocks];
    for (int w = 0; w < NW; ++w) {
      const int i = split * kSplitBlocks + w;
      bl[w] = -1;
      if (i < K) {
        const int e = selrow[i];
        const int prev = i > 0 ? selrow[i - 1] : -1;
        if (e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e))) bl[w] = e;
      }
      if (bl[w] >= 0) total += 2u * kBlockElems * 2u;
    }
    mbar_arrive_expect_tx(&bar, total);
    for (int w = 0; w < NW; ++w) {
      if (bl[w] < 0) continue;
      const int64_t row = row_of(a, s, h, bl[w]);
      bulk_g2s(kv_smem + (size_t)w * 2 * kBlockElems, a.k + row * kBlockElems, kBlockElems * 2u, &bar);
      bulk_g2s(kv_smem + (size_t)w * 2 * kBlockElems + kBlockElems, a.v + row * kBlockElems, kBlockElems * 2u,
               &bar);
    }
  }

  float qr[G][V];
  const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) qr[g][i] = qg[g * D + lane * V + i] * InvSqrtDA<D>::v;
  float m[G], l[G], acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  }

  // compensation sums of the scoring items assigned to this work item
  if (comp) {
    const int c0 = (int)((int64_t)split * nch / a.splits), c1 = (int)((int64_t)(split + 1) * nch / a.splits);
    const int rs = rec_stride(a);
    for (int c = c0 + warp; c < c1; c += NW) {
      const float* rec = a.chunk_rec + (int64_t)(rec0 + c) * rs;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mc = __ldcg(rec + g * (4 + D) + 2);
        const float lc = __ldcg(rec + g * (4 + D) + 3);
        float fo, fn;
        rescale_to(m[g], mc, fo, fn);
        l[g] = l[g] * fo + lc * fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo + __ldcg(rec + g * (4 + D) + 4 + lane * V + i) * fn;
      }
    }
  }

  mbar_wait_bounded(&bar, 0, a.status, s, h, 31);
  __syncthreads();

  if (my_b >= 0) {
    const int n = (my_b == N - 1) ? L - kBlock * my_b : kBlock;
    const __nv_bfloat16* ks = kv_smem + (size_t)warp * 2 * kBlockElems;
    const __nv_bfloat16* vs = ks + kBlockElems;
    float z[G][kBlock];
#pragma unroll
    for (int j = 0; j < kBlock; ++j) {
      float kf[V];
      load_bf16<V>(ks + j * D + lane * V, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) t = fmaf(qr[g][i], kf[i], t);
        z[g][j] = t;
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int j = 0; j < kBlock; ++j) z[g][j] = warp_sum(z[g][j]);
    }
    float bm[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      bm[g] = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBlock; ++j)
        if (j < n) bm[g] = fmaxf(bm[g], z[g][j]);
      float fo, fn;
      rescale_to(m[g], bm[g], fo, fn);
      l[g] *= fo;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[g][i] *= fo;
    }
#pragma unroll
    for (int j = 0; j < kBlock; ++j) {
      if (j < n) {
        float vf[V];
        load_bf16<V>(vs + j * D + lane * V, vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = expf(z[g][j] - m[g]);
          l[g] += p;
#pragma unroll
          for (int i = 0; i < V; ++i) acc[g][i] = fmaf(p, vf[i], acc[g][i]);
        }
      }
    }
    if (comp) {
      // remove this block's Mean compensation term (it was added for every block)
      const int c = my_b / kChunk, o = my_b % kChunk;
      const float lnn = ln_count_a(n);
      const int64_t row = row_of(a, s, h, my_b);
      float vb[V];
#pragma unroll
      for (int i = 0; i < V; ++i) vb[i] = __ldcg(a.vbar + row * D + lane * V + i);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float e = lnn + __ldcg(a.chunk_z + ((int64_t)(rec0 + c) * G + g) * kChunk + o);
        float fo, fn;
        rescale_to(m[g], e, fo, fn);
        l[g] = l[g] * fo - fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo - fn * vb[i];
      }
    }
  }

  // merge the warps
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp][g] = m[g];
      red_l[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < V; ++i) red_acc[warp][g][lane * V + i] = acc[g][i];
  }
  __syncthreads();
  float* srec = a.split_rec + ((int64_t)sh * a.splits + split) * rec_stride(a);
  for (int idx = tid; idx < G * D; idx += 256) {
    const int g = idx / D, col = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w][g]);
    float ls = 0.f, as = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = (red_m[w][g] == -INFINITY) ? 0.f : expf(red_m[w][g] - M);
        ls += red_l[w][g] * f;
        as += red_acc[w][g][col] * f;
      }
    }
    if (col == 0) {
      srec[g * (4 + D) + 0] = M;
      srec[g * (4 + D) + 1] = ls;
    }
    srec[g * (4 + D) + 4 + col] = as;
  }
  // the last work item of this (sequence, head) merges all of them
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(a.head_counter + sh, 1);
    sh_last = (prev == a.splits - 1);
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  const float* recs = a.split_rec + (int64_t)sh * a.splits * rec_stride(a);
  float* out = a.out + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
  for (int idx = tid; idx < G * D; idx += 256) {
    const int g = idx / D, col = idx % D;
    float M = -INFINITY;
    for (int p = 0; p < a.splits; ++p) M = fmaxf(M, __ldcg(recs + (int64_t)p * rec_stride(a) + g * (4 + D)));
    float ls = 0.f, as = 0.f;
    if (M != -INFINITY) {
      for (int p = 0; p < a.splits; ++p) {
        const float* rp = recs + (int64_t)p * rec_stride(a) + g * (4 + D);
        const float mp = __ldcg(rp);
        const float f = (mp == -INFINITY) ? 0.f : expf(mp - M);
        ls += __ldcg(rp + 1) * f;
        as += __ldcg(rp + 4 + col) * f;
      }
    }
    out[g * D + col] = (ls > 0.f) ? as / ls : 0.f;
  }
  if (tid == 0) a.head_counter[sh] = 0;
}

template <int D, int G>
static cudaError_t launch_attend_dg(const LayerArgs& a, cudaStream_t st) {
  const size_t sm = (size_t)8 * 2 * kBlock * D * sizeof(__nv_bfloat16);
  cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  attend_kernel<D, G><<<a.B * a.Hkv * a.splits, 256, sm, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attend(const LayerArgs& a, cudaStream_t st) {
#define COMPKV_G(DD)                                      \
  switch (a.G) {                                          \
    case 1: return launch_attend_dg<DD, 1>(a, st);        \
    case 2: return launch_attend_dg<DD, 2>(a, st);        \
    case 4: return launch_attend_dg<DD, 4>(a, st);        \
    case 8: return launch_attend_dg<DD, 8>(a, st);        \
    default: return cudaErrorInvalidValue;                \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

}  // namespace compkv
