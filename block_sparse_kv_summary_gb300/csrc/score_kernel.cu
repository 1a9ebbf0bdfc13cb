// Scoring pass over the block summaries (CompKV, section "무엇과 다른가").
//
// One CTA per work item = up to 64 consecutive blocks of one (sequence, KV
// head).  A single thread stages the item's kbar (and vbar, Dbar) rows into
// shared memory with 1-D bulk copies completing on an mbarrier; the CTA then
//   pass 1  zbar_{g,b} = q_g . kbar_b / sqrt(d) and
//           sigma2_{g,b} = (1/d) sum_t Qsq_{g,t} (Dbar_b)_t, Qsq_{g,t} = sum_{i in G_t} q_{g,i}^2
//           (16 lanes per block, reduced with shuffles),
//   pass 2  a_{g,b} = ln|b| + zbar + sigma2/2; per query head the item's
//           max m_a and sum exp(a - m_a) (its share of the logsumexp that
//           normalises the mass estimate), and u_{g,b} = exp(a - m_a) sigma2
//           so that phat_{g,b} sigma2_{g,b} = u_{g,b} exp(m_a - LSE_g);
//           for Mean compensation the weights w_{g,b} = exp(ln|b| + zbar - m_c),
//   pass 3  sum_b w_{g,b} vbar_b (the item's share of the compensation of
//           every block; the selected ones are subtracted after selection).
// Everything is fp32.  The per-item records are small and stay in L2.
#include "compkv_launch.h"

namespace compkv {

template <int D>
struct InvSqrtD;
template <>
struct InvSqrtD<64> {
  static constexpr float v = 0.125f;
};
template <>
struct InvSqrtD<128> {
  static constexpr float v = 0.08838834764831845f;
};

__device__ __forceinline__ float ln_count(int n) { return n == kBlock ? 2.772588722239781f : logf((float)n); }

struct ScoreSmem {
  // offsets in floats
  int k, v, dbar, q, qsq, z, s2, w, bar_off_bytes, total_bytes;
};

__host__ __device__ inline ScoreSmem score_layout(int D, int r, int G, int mode) {
  ScoreSmem L;
  int off = 0;
  L.k = off;
  off += kChunk * D;
  L.v = off;
  if (mode & kModeComp) off += kChunk * D;
  L.dbar = off;
  if (mode & kModeScore) off += kChunk * r;
  off = (off + 3) & ~3;
  L.q = off;
  off += G * D;
  L.qsq = off;
  off += ((G * r + 3) & ~3);
  L.z = off;
  off += G * kChunk;
  L.s2 = off;
  off += G * kChunk;
  L.w = off;
  off += G * kChunk;
  L.bar_off_bytes = ((off * 4) + 15) & ~15;
  L.total_bytes = L.bar_off_bytes + 16;
  return L;
}

size_t score_smem_bytes(int d, int r, int G, int mode) { return (size_t)score_layout(d, r, G, mode).total_bytes; }

template <int D, int G, int MODE>
__global__ void __launch_bounds__(256) score_kernel(LayerArgs a) {
  constexpr bool SCORE = (MODE & kModeScore) != 0;
  constexpr bool COMP = (MODE & kModeComp) != 0;
  constexpr int NT = 256;
  constexpr int NW = NT / 32;
  extern __shared__ __align__(128) float smem[];

  const int rec = blockIdx.x;
  int s = 0;
  while (s + 1 < a.B && a.chunk0[s + 1] <= rec) ++s;
  const int local = rec - a.chunk0[s];
  const int h = local / a.nchunk[s];
  const int c = local % a.nchunk[s];
  const int L = seq_tokens(a, s);
  const int N = ceil_blocks(L);
  const int b0 = c * kChunk;
  if (h >= a.Hkv || b0 >= N) return;
  const int nb = min(kChunk, N - b0);
  const int r = a.r;
  const int64_t row0 = row_of(a, s, h, b0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const ScoreSmem lay = score_layout(D, r, G, MODE);
  float* sk = smem + lay.k;
  float* sv = smem + lay.v;
  float* sd = smem + lay.dbar;
  float* sq = smem + lay.q;
  float* sqsq = smem + lay.qsq;
  float* sz = smem + lay.z;
  float* ss = smem + lay.s2;
  float* sw = smem + lay.w;
  uint64_t* bar = reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(smem) + lay.bar_off_bytes);
  const bool dbar_bulk = SCORE && ((r & 3) == 0);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t bytes = (uint32_t)nb * D * 4u;
    uint32_t total = bytes;
    if (COMP) total += bytes;
    if (dbar_bulk) total += (uint32_t)nb * r * 4u;
    mbar_arrive_expect_tx(bar, total);
    bulk_g2s(sk, a.kbar + row0 * D, bytes, bar);
    if (COMP) bulk_g2s(sv, a.vbar + row0 * D, bytes, bar);
    if (dbar_bulk) bulk_g2s(sd, a.dbar + row0 * r, (uint32_t)nb * r * 4u, bar);
  }
  // queries of this GQA group and their grouped squared norms
  const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
  for (int i = tid; i < G * D; i += NT) sq[i] = qg[i];
  if (SCORE && !dbar_bulk)
    for (int i = tid; i < nb * r; i += NT) sd[i] = a.dbar[row0 * r + i];
  __syncthreads();
  if (SCORE) {
    const int gs = D / r;
    for (int i = tid; i < G * r; i += NT) {
      const int g = i / r, t = i % r;
      float acc = 0.f;
      for (int j = 0; j < gs; ++j) {
        const float x = sq[g * D + t * gs + j];
        acc = fmaf(x, x, acc);
      }
      sqsq[i] = acc;
    }
  }
  mbar_wait_bounded(bar, 0, a.status, s, h, 10);
  __syncthreads();

  // ---- pass 1: 16 lanes per block; lane j holds coordinates {4j..4j+3} (+64 at D = 128)
  {
    constexpr int NV4 = D / 64;  // float4s per lane
    const int hw = tid >> 4, j = tid & 15;
    float qr[G][NV4 * 4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int u = 0; u < NV4; ++u) {
        const float4 t = *reinterpret_cast<const float4*>(sq + g * D + u * 64 + 4 * j);
        qr[g][4 * u + 0] = t.x;
        qr[g][4 * u + 1] = t.y;
        qr[g][4 * u + 2] = t.z;
        qr[g][4 * u + 3] = t.w;
      }
    // the loop bound is uniform per warp (the two half-warps share every trip),
    // so the full-mask shuffles below always see all 32 lanes
    for (int base = warp * 2; base < nb; base += NT / 16) {
      const int blk = base + (hw & 1);
      const bool valid = blk < nb;
      const int rb = valid ? blk : base;
      float zacc[G], sacc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) zacc[g] = sacc[g] = 0.f;
#pragma unroll
      for (int u = 0; u < NV4; ++u) {
        const float4 kv = *reinterpret_cast<const float4*>(sk + rb * D + u * 64 + 4 * j);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          zacc[g] = fmaf(qr[g][4 * u + 0], kv.x, zacc[g]);
          zacc[g] = fmaf(qr[g][4 * u + 1], kv.y, zacc[g]);
          zacc[g] = fmaf(qr[g][4 * u + 2], kv.z, zacc[g]);
          zacc[g] = fmaf(qr[g][4 * u + 3], kv.w, zacc[g]);
        }
      }
      if (SCORE) {
        for (int t = j; t < r; t += 16) {
          const float dv = sd[rb * r + t];
#pragma unroll
          for (int g = 0; g < G; ++g) sacc[g] = fmaf(sqsq[g * r + t], dv, sacc[g]);
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          zacc[g] += __shfl_xor_sync(0xffffffffu, zacc[g], o);
          if (SCORE) sacc[g] += __shfl_xor_sync(0xffffffffu, sacc[g], o);
        }
      }
      if (j == 0 && valid) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          sz[g * kChunk + blk] = zacc[g] * InvSqrtD<D>::v;
          if (SCORE) ss[g * kChunk + blk] = sacc[g] / (float)D;
        }
      }
    }
  }
  __syncthreads();

  // ---- pass 2: one warp per query head
  float* recp = a.chunk_rec + (int64_t)rec * rec_stride(a);
  if (warp < G) {
    const int g = warp;
    float av[kChunk / 32], cv[kChunk / 32];
    float ma = -INFINITY, mc = -INFINITY;
#pragma unroll
    for (int i = 0; i < kChunk / 32; ++i) {
      const int blk = lane + 32 * i;
      av[i] = cv[i] = -INFINITY;
      if (blk < nb) {
        const int bb = b0 + blk;
        const int n = (bb == N - 1) ? L - kBlock * bb : kBlock;
        const float lnn = ln_count(n);
        const float z = sz[g * kChunk + blk];
        cv[i] = lnn + z;
        if (SCORE) av[i] = cv[i] + 0.5f * ss[g * kChunk + blk];
      }
      ma = fmaxf(ma, av[i]);
      mc = fmaxf(mc, cv[i]);
    }
    float la = 0.f, lc = 0.f;
    if (SCORE) {
      ma = warp_max(ma);
#pragma unroll
      for (int i = 0; i < kChunk / 32; ++i) {
        const int blk = lane + 32 * i;
        const float e = (blk < nb) ? expf(av[i] - ma) : 0.f;
        la += e;
        a.chunk_u[((int64_t)rec * G + g) * kChunk + blk] = (blk < nb) ? e * ss[g * kChunk + blk] : 0.f;
      }
      la = warp_sum(la);
    }
    if (COMP) {
      mc = warp_max(mc);
#pragma unroll
      for (int i = 0; i < kChunk / 32; ++i) {
        const int blk = lane + 32 * i;
        const float w = (blk < nb) ? expf(cv[i] - mc) : 0.f;
        lc += w;
        sw[g * kChunk + blk] = w;
        a.chunk_z[((int64_t)rec * G + g) * kChunk + blk] = (blk < nb) ? sz[g * kChunk + blk] : 0.f;
      }
      lc = warp_sum(lc);
    }
    if (lane == 0) {
      float* rg = recp + g * (4 + D);
      rg[0] = ma;
      rg[1] = la;
      rg[2] = mc;
      rg[3] = lc;
    }
  }

  // ---- pass 3: compensation numerator sum_b w_{g,b} vbar_b
  if (COMP) {
    __syncthreads();
    constexpr int V = D / 32;
    float acc[G][V];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
    for (int blk = warp; blk < nb; blk += NW) {
      float vv[V];
      if (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(sv + blk * D + lane * 4);
        vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(sv + blk * D + lane * 2);
        vv[0] = t.x; vv[1] = t.y;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w = sw[g * kChunk + blk];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = fmaf(w, vv[i], acc[g][i]);
      }
    }
    // cross-warp reduction through the (now free) kbar staging area
    float* red = sk;  // [NW][G][D]
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < V; ++i) red[(warp * G + g) * D + lane * V + i] = acc[g][i];
    __syncthreads();
    for (int i = tid; i < G * D; i += NT) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) t += red[w * G * D + i];
      const int g = i / D, col = i % D;
      recp[g * (4 + D) + 4 + col] = t;
    }
  }
}

template <int D, int G>
static cudaError_t launch_score_dg(const LayerArgs& a, int mode, int total, cudaStream_t st) {
  const size_t sm = score_smem_bytes(D, a.r, G, mode);
  cudaError_t e = cudaSuccess;
#define COMPKV_SCORE_CASE(M)                                                                           \
  case M:                                                                                              \
    e = cudaFuncSetAttribute(score_kernel<D, G, M>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm); \
    if (e != cudaSuccess) return e;                                                                    \
    score_kernel<D, G, M><<<total, 256, sm, st>>>(a);                                                  \
    break;
  switch (mode) {
    COMPKV_SCORE_CASE(1)
    COMPKV_SCORE_CASE(2)
    COMPKV_SCORE_CASE(3)
    default:
      return cudaErrorInvalidValue;
  }
#undef COMPKV_SCORE_CASE
  return cudaGetLastError();
}

cudaError_t launch_score(const LayerArgs& a, int mode, int total_records, cudaStream_t st) {
  if (total_records <= 0) return cudaSuccess;
#define COMPKV_G(DD)                                                \
  switch (a.G) {                                                    \
    case 1: return launch_score_dg<DD, 1>(a, mode, total_records, st); \
    case 2: return launch_score_dg<DD, 2>(a, mode, total_records, st); \
    case 4: return launch_score_dg<DD, 4>(a, mode, total_records, st); \
    case 8: return launch_score_dg<DD, 8>(a, mode, total_records, st); \
    default: return cudaErrorInvalidValue;                          \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

}  // namespace compkv
