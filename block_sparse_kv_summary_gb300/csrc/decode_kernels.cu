// The CompKV decode step (onedev.kr/papers/157) as three kernels chained with
// programmatic dependent launch.
//
// Section "무엇과 다른가" of the CompKV page defines the step per (sequence,
// KV head) "unit": score every 16-token block from its summary, select the
// sink block, the two most recent blocks and the Top-K of S_b, attend exactly
// to the selected blocks and add Mean compensation for the others under one
// normaliser.  Section "어떻게 쓰나" fuses the open block's summary update
// with the K/V pack; here that happens in the first kernel.
//
//   1. score   one CTA per item of 64 blocks: kbar, Dbar and the unit's
//              queries staged by 1-D bulk copies (cp.async.bulk, mbarrier) in
//              two halves; zbar = q.kbar/sqrt(d), sigma2 = (1/d) sum_t
//              Qsq_t Dbar_t, a = ln|b| + zbar + sigma2/2; per query head the
//              item's max a, sum e^(a - max a), max(ln|b| + zbar), and per
//              block u = e^(a - max a) sigma2 and zbar.  The item holding the
//              newest token appends it first.
//   2. S items     one CTA per 512 blocks of a unit: LSE_g from the scoring
//              records, S_b = sum_g u e^(max a - LSE_g) = sum_g phat sigma2 as
//              order-preserving keys, their exponent histogram; the unit's
//              last S item selects: forced set + the K-3 largest S_b by an
//              exponent-first radix select (ties to the lower index).
//      comp items  in the same grid, one CTA per 128 blocks of a unit: their
//              vbar rows (bulk-copied before the dependency wait, overlapping
//              the scoring kernel's tail) weighted by w = e^(ln|b| + zbar -
//              M_g), M_g = max_b (ln|b| + zbar), summed into the unit's
//              accumulator (fp32 atomics) -- over every block.
//   3. attend  one CTA per 8 selected blocks: exact softmax terms of their
//              tokens (one block per warp), minus each selected block's own
//              compensation term (it was summed for every block in 2), as a
//              partial (m, l, acc); the last CTA of the unit merges the
//              partials with the compensation sum into out = acc / l.
// By Jensen, sum_{j in b} e^{z_j} >= |b| e^{zbar_b}, so removing a selected
// block's mean term never makes a denominator negative.  If every block is
// selected the compensation is skipped (the step is dense attention).
#include <atomic>

#include "compkv_launch.h"

namespace compkv {

constexpr int kT = 256;            // threads per CTA, all three kernels
constexpr int kW = kT / 32;
constexpr int kPrivBins = 256;     // histogram bins of one radix digit
constexpr int kListMax = 2048;     // keys in play compacted into a list once at most this many
constexpr int kRankMax = 512;      // listed keys in play ranked directly once at most this many
constexpr int kChunkS = 8 * kChunk;  // blocks per S item

template <int D>
struct InvSqrt;
template <>
struct InvSqrt<64> {
  static constexpr float v = 0.125f;
};
template <>
struct InvSqrt<128> {
  static constexpr float v = 0.08838834764831845f;
};

__device__ __forceinline__ float ln_n(int n) { return n == kBlock ? 2.772588722239781f : logf((float)n); }

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Tokens of sequence s in this call (after its append when `append`).
__device__ __forceinline__ int unit_tokens(const LayerArgs& a, int s, bool append, bool* fits) {
  const int Lold = a.seq_len[s];
  const int cap = a.cap_blocks[s] * kBlock;
  *fits = Lold >= 0 && Lold < cap;
  int L = Lold < 0 ? 0 : (Lold > cap ? cap : Lold);
  if (append && *fits) L += 1;
  return L;
}

__device__ __forceinline__ int chunk_record(const LayerArgs& a, int s, int h, int c) {
  return a.chunk0[s] + h * a.nchunk[s] + c;
}

// Trace slots: scoring CTAs, S items, compensation items, one selection record
// per unit, attention CTAs, then 32 phase marks per unit.
__device__ __forceinline__ int slot_items(const LayerArgs& a) { return a.total_chunks; }
__device__ __forceinline__ int slot_select(const LayerArgs& a) { return a.total_chunks + a.ns_items + a.n2_items; }
__device__ __forceinline__ int slot_attend(const LayerArgs& a) { return slot_select(a) + a.B * a.Hkv; }
__device__ __forceinline__ int slot_phase(const LayerArgs& a) { return slot_attend(a) + a.B * a.Hkv * a.splits; }

// Record (cta << 32 | type << 24 | index), unit, t0, t1, now, x0, x1, x2 into `slot`.
__device__ __forceinline__ void trace_item(const LayerArgs& a, int slot, int type, int unit, int index,
                                           unsigned long long t0, unsigned long long t1, unsigned long long x0 = 0,
                                           unsigned long long x1 = 0, unsigned long long x2 = 0) {
  if (!a.trace || slot < 0 || slot >= a.trace_cap) return;
  const unsigned long long now = global_ns();
  unsigned long long* r = a.trace + 1 + 8 * (int64_t)slot;
  r[0] = ((unsigned long long)blockIdx.x << 32) | ((unsigned long long)(type & 0xff) << 24) | (unsigned)(index & 0xffffff);
  r[1] = (unsigned long long)unit;
  r[2] = t0;
  r[3] = t1;
  r[4] = now;
  r[5] = x0;
  r[6] = x1;
  r[7] = x2;
}

// Phase mark k (< 16) of unit u's selection (trace type 5, index = phase): from `t_prev` to now.
__device__ __forceinline__ unsigned long long trace_phase(const LayerArgs& a, int unit, int k, int phase,
                                                          unsigned long long t_prev) {
  if (!a.trace) return 0ull;
  const unsigned long long now = global_ns();
  trace_item(a, slot_phase(a) + unit * 32 + (k & 15), 5, unit, phase, t_prev, now);
  return now;
}

// ================================================================== 1. score
// Lane layout: lane = g * LPG + p; lane p of query head g holds coordinates
// [p * DPL, (p + 1) * DPL) of q_g in 4-wide chunks, chunk i of the lane at
// position (i + p) mod NCH so that the LPG lanes reading one kbar row touch
// different banks.  A block costs a lane DPL FMAs for zbar and a few for
// sigma2, then log2(LPG) butterfly steps.
template <int D, int G>
struct ScoreLayout {
  static constexpr int LPG = 32 / G;         // lanes per query head
  static constexpr int DPL = D / LPG;        // coordinates per lane (>= 2)
  static constexpr int CW = DPL >= 4 ? 4 : DPL;
  static constexpr int NCH = DPL / CW;       // chunks per lane
};

// shared memory: kbar rows | Dbar rows | variance scratch (D) | zbar, sigma2 | Qsq (G x r, padded
// to 4) | 2 mbarriers
__host__ __device__ inline int score_smem(int D, int r, int G) {
  return (kChunk * (D + r) + D + 2 * G * kChunk + ((G * r + 3) & ~3)) * 4 + 32;
}

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kT, 4) k_score(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  using SL = ScoreLayout<D, G>;
  constexpr int LPG = SL::LPG, DPL = SL::DPL, CW = SL::CW, NCH = SL::NCH;
  extern __shared__ __align__(128) float sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  int s = 0;
  while (s + 1 < a.B && a.chunk0[s + 1] <= (int)blockIdx.x) ++s;
  const int local = blockIdx.x - a.chunk0[s];
  const int h = local / a.nchunk[s], c = local % a.nchunk[s];
  const int u = s * a.Hkv + h;
  const int r = a.r;
  pdl_wait();  // the previous work on the stream may have written this cache
  const unsigned long long t_pdl = a.trace ? global_ns() : 0ull;
  bool fits;
  const int L = unit_tokens(a, s, APPEND, &fits);
  const int N = ceil_blocks(L);
  if (blockIdx.x == 0 && tid < a.B) {
    bool f2;
    a.lnew[tid] = unit_tokens(a, tid, APPEND, &f2);
  }
  if (COMP && c == 0)
    for (int i = tid; i < G * (D + 4); i += kT) a.unit_acc[(int64_t)u * G * (D + 4) + i] = 0.f;
  pdl_trigger();
  const int b0 = c * kChunk;
  if (b0 >= N) return;
  const int nb = min(kChunk, N - b0);
  const bool append = APPEND && fits && b0 + nb == N;
  const int nt = nb - (append ? 1 : 0);  // rows copied from global memory
  const int rec = chunk_record(a, s, h, c);
  float* sk = sm;
  float* sd = sk + kChunk * D;
  float* svar = sd + kChunk * r;
  float* zs = svar + D;
  float* ss = zs + G * kChunk;
  float* sqs = ss + G * kChunk;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sqs + ((G * r + 3) & ~3));
  const int64_t row0 = row_of(a, s, h, b0);
  const bool dbar_bulk = SCORE && (r & 3) == 0;
  constexpr int kHalf = kChunk / 2;
  const int nA = min(nt, kHalf), nB = nt - nA;
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
    const uint32_t rowb = (uint32_t)D * 4u + (dbar_bulk ? (uint32_t)r * 4u : 0u);
    mbar_arrive_expect_tx(bar, (uint32_t)nA * rowb);
    if (nA > 0) {
      bulk_g2s(sk, a.kbar + row0 * D, (uint32_t)nA * D * 4u, bar);
      if (dbar_bulk) bulk_g2s(sd, a.dbar + row0 * r, (uint32_t)nA * r * 4u, bar);
    }
    mbar_arrive_expect_tx(bar + 1, (uint32_t)nB * rowb);
    if (nB > 0) {
      bulk_g2s(sk + kHalf * D, a.kbar + (row0 + kHalf) * D, (uint32_t)nB * D * 4u, bar + 1);
      if (dbar_bulk) bulk_g2s(sd + kHalf * r, a.dbar + (row0 + kHalf) * r, (uint32_t)nB * r * 4u, bar + 1);
    }
  }
  // this lane's slice of q_g straight from global memory (L2), while the rows land
  const int g = lane / LPG, p = lane % LPG;
  const float* qg_glob = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G + g) * D;
  float qr[NCH][CW];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int cpos = p * DPL + CW * ((i + p) & (NCH - 1));
    if (CW == 4) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(qg_glob + cpos));
      qr[i][0] = x.x;
      qr[i][1 % CW] = x.y;
      qr[i][2 % CW] = x.z;
      qr[i][3 % CW] = x.w;
    } else {
      const float2 x = __ldg(reinterpret_cast<const float2*>(qg_glob + cpos));
      qr[i][0] = x.x;
      qr[i][1 % CW] = x.y;
    }
  }
  if (SCORE && (r & 3))
    for (int i = tid; i < nt * r; i += kT) sd[i] = a.dbar[row0 * r + i];
  if (append) {
    // pack the new token and recompute the open block's summary from its
    // tokens: thread c < D owns key coordinate c, thread D + c value
    // coordinate c; mean and population variance two-pass in fp32 from the
    // exact bf16 values (no E[k^2] - E[k]^2 cancellation)
    const int n = L - kBlock * (N - 1);
    const int64_t row = row0 + (nb - 1);
    if (tid < 2 * D) {
      const bool isk = tid < D;
      const int cc = isk ? tid : tid - D;
      const __nv_bfloat16* src = (isk ? a.k : a.v) + row * kBlock * D + cc;
      const __nv_bfloat16 xn = (isk ? a.k_new : a.v_new)[((int64_t)s * a.Hkv + h) * D + cc];
      float x[kBlock];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < kBlock; ++j) {
        x[j] = 0.f;
        if (j < n - 1) x[j] = __bfloat162float(src[j * D]);
        if (j == n - 1) x[j] = __bfloat162float(xn);
        sum += x[j];
      }
      (isk ? a.k : a.v)[(row * kBlock + n - 1) * D + cc] = xn;
      const float mean = sum / (float)n;
      if (isk) {
        float var = 0.f;
#pragma unroll
        for (int j = 0; j < kBlock; ++j)
          if (j < n) var = fmaf(x[j] - mean, x[j] - mean, var);
        sk[(nb - 1) * D + cc] = mean;
        a.kbar[row * D + cc] = mean;
        svar[cc] = var / (float)n;
      } else {
        a.vbar[row * D + cc] = mean;
      }
    }
    __syncthreads();
    if (tid < r) {
      // Dbar_t: mean of the variances over coordinate group t = [t*D/r, (t+1)*D/r)
      const int gs = D / r;
      float t = 0.f;
      for (int i = 0; i < gs; ++i) t += svar[tid * gs + i];
      t /= (float)gs;
      sd[(nb - 1) * r + tid] = t;
      a.dbar[row * r + tid] = t;
    }
  }
  __syncthreads();
  mbar_wait_bounded(bar, 0, a.status, s, h, 10);
  const unsigned long long t_a = a.trace ? global_ns() : 0ull;
  // ---- zbar and sigma2: one block per warp at a time, query heads on lanes
  // sigma2 weights: lanes whose coordinates lie in one group t (r <= LPG)
  // weight Dbar_t by their sum of q^2; otherwise lane p takes the groups
  // [p * rpl, (p + 1) * rpl), rotated like the kbar chunks, with Qsq_{g,t}
  // from shared memory
  const int gs = D / r;
  const bool one_group = r <= LPG;
  const int rpl = one_group ? 1 : r / LPG;
  const int t_one = (p * DPL) / gs;
  float qsq_one = 0.f;
#pragma unroll
  for (int i = 0; i < NCH; ++i)
#pragma unroll
    for (int j = 0; j < CW; ++j) qsq_one = fmaf(qr[i][j], qr[i][j], qsq_one);
  if (SCORE && !one_group) {
    for (int i = tid; i < G * r; i += kT) {
      const float* qp = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G + i / r) * D + (i % r) * gs;
      float t = 0.f;
      for (int k = 0; k < gs; ++k) t = fmaf(qp[k], qp[k], t);
      sqs[i] = t;
    }
    __syncthreads();
  }
  auto do_block = [&](int blk) {
    const float* krow = sk + blk * D + p * DPL;
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      const int off = CW * ((i + p) & (NCH - 1));
      if (CW == 4) {
        const float4 x = *reinterpret_cast<const float4*>(krow + off);
        z = fmaf(qr[i][0], x.x, z);
        z = fmaf(qr[i][1 % CW], x.y, z);
        z = fmaf(qr[i][2 % CW], x.z, z);
        z = fmaf(qr[i][3 % CW], x.w, z);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(krow + off);
        z = fmaf(qr[i][0], x.x, z);
        z = fmaf(qr[i][1 % CW], x.y, z);
      }
    }
    float sg = 0.f;
    if (SCORE) {
      const float* drow = sd + blk * r;
      if (one_group) {
        sg = qsq_one * drow[t_one];
      } else {
        const float* qrow = sqs + g * r + p * rpl;
        const float* dseg = drow + p * rpl;
        for (int k = 0; k < rpl; ++k) {
          const int t = (k + p) & (rpl - 1);
          sg = fmaf(qrow[t], dseg[t], sg);
        }
      }
    }
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) {
      z += __shfl_xor_sync(0xffffffffu, z, o);
      if (SCORE) sg += __shfl_xor_sync(0xffffffffu, sg, o);
    }
    if (p == 0) {
      zs[g * kChunk + blk] = z * InvSqrt<D>::v;
      if (SCORE) ss[g * kChunk + blk] = sg / (float)D;
    }
  };
#pragma unroll
  for (int it = 0; it < kHalf / kW; ++it) {
    const int blk = warp + kW * it;
    if (blk < nb) do_block(blk);
  }
  const unsigned long long t_b = a.trace ? global_ns() : 0ull;
  if (nb > kHalf) {
    mbar_wait_bounded(bar + 1, 0, a.status, s, h, 13);
#pragma unroll
    for (int it = kHalf / kW; it < kChunk / kW; ++it) {
      const int blk = warp + kW * it;
      if (blk < nb) do_block(blk);
    }
  }
  const unsigned long long t_loaded = a.trace ? global_ns() : 0ull;
  __syncthreads();
  // ---- per query head: item max and sum of e^a, u per block, max of ln|b| + zbar
  if (warp < G) {
    const int gw = warp;
    float av[2], cv[2];
    float ma = -INFINITY, mc = -INFINITY;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int blk = lane + 32 * i;
      av[i] = cv[i] = -INFINITY;
      if (blk < nb) {
        const int bb = b0 + blk;
        const int n = (bb == N - 1) ? L - kBlock * bb : kBlock;
        cv[i] = ln_n(n) + zs[gw * kChunk + blk];
        if (SCORE) av[i] = cv[i] + 0.5f * ss[gw * kChunk + blk];
      }
      ma = fmaxf(ma, av[i]);
      mc = fmaxf(mc, cv[i]);
    }
    mc = warp_max(mc);
    float la = 0.f;
    if (SCORE) {
      ma = warp_max(ma);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int blk = lane + 32 * i;
        const float e = (blk < nb) ? expf(av[i] - ma) : 0.f;
        la += e;
        a.chunk_u[((int64_t)rec * G + gw) * kChunk + blk] = (blk < nb) ? e * ss[gw * kChunk + blk] : 0.f;
      }
      la = warp_sum(la);
    }
    if (COMP) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int blk = lane + 32 * i;
        a.chunk_z[((int64_t)rec * G + gw) * kChunk + blk] = (blk < nb) ? zs[gw * kChunk + blk] : 0.f;
      }
    }
    if (lane == 0)
      *reinterpret_cast<float4*>(a.chunk_rec + ((int64_t)rec * G + gw) * 4) = make_float4(ma, la, mc, 0.f);
  }
  if (tid == 0) trace_item(a, blockIdx.x, 0, u, c, t_start, t_loaded, t_pdl, t_a, t_b);
}

// ================================================================== 2. S items, selection, compensation
// Shared memory of the grid (the larger of the two item kinds):
//   S item:    selection region (keys | per-warp histograms | summed
//              histogram | list keys | list indices | bitmap | prefix) |
//              item factors (8 x G) | histogram (256) | misc (32)
//   comp item: vbar rows (128 x D) | weights (G x 128) | M_g (G) | mbarrier
__host__ __device__ inline int sel_region_words(int key_stride) {
  const int words = (key_stride + 31) / 32 + 4;
  return key_stride + 4 + (kW + 1) * kPrivBins + 2 * (kListMax + 4) + 2 * words;
}
__host__ __device__ inline int s_item_smem(int G, int key_stride) {
  return (((sel_region_words(key_stride) + 3) & ~3) + 8 * G + kPrivBins + 32) * 4;
}
__host__ __device__ inline int comp_bar_offset(int D, int G) { return ((kChunk2 * D + G * kChunk2 + G) * 4 + 15) & ~15; }
__host__ __device__ inline int comp_item_smem(int D, int G) { return comp_bar_offset(D, G) + 16; }
__host__ __device__ inline int item_grid_smem(int D, int G, int key_stride, bool sel, bool comp) {
  int m = 0;
  if (sel) m = s_item_smem(G, key_stride);
  if (comp && comp_item_smem(D, G) > m) m = comp_item_smem(D, G);
  return m;
}

// Warp 0: wbase[w] = set bits in words[0..w), for w < nw; returns the total
// (in warp 0; other warps get 0).
__device__ __forceinline__ int word_prefix(const unsigned* words, int* wbase, int nw, int lane, int warp) {
  if (warp != 0) return 0;
  const int per = (nw + 31) / 32;
  int loc = 0;
  for (int i = 0; i < per; ++i) {
    const int w = per * lane + i;
    if (w < nw) loc += __popc(words[w]);
  }
  int incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - loc;
  for (int i = 0; i < per; ++i) {
    const int w = per * lane + i;
    if (w < nw) {
      wbase[w] = run;
      run += __popc(words[w]);
    }
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// Warp 0 over a histogram of nbins (256 or 128) digits, scanned from the top:
// misc[0] = the digit at which the count of larger-or-equal keys reaches
// `need`, misc[1] = keys above it, misc[2] = keys at it.  Ends with a CTA barrier.
__device__ __forceinline__ void find_digit(const uint32_t* hh, int nbins, int need, int* misc, int lane, int warp) {
  if (warp == 0) {
    const int per = nbins / 32;
    uint32_t cnt[8];
    int loc = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cnt[i] = i < per ? hh[nbins - 1 - per * lane - i] : 0u;
      loc += (int)cnt[i];
    }
    int incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int before = incl - loc;
    if (before < need && need <= incl) {
      int run = before;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < per && run < need && need <= run + (int)cnt[i]) {
          misc[0] = nbins - 1 - per * lane - i;
          misc[1] = run;
          misc[2] = (int)cnt[i];
        }
        run += (int)cnt[i];
      }
    }
  }
  __syncthreads();
}

// Exclusive prefix of `v` over the CTA (`scratch`: kW ints); every thread
// gets its offset; `total` receives the sum.  Contains two CTA barriers.
__device__ __forceinline__ int cta_exclusive_scan(int v, int* scratch, int* total, int lane, int warp) {
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const int t = scratch[w];
    base += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// Selection for unit u by its last S item: the unit's keys (S_b as
// order-preserving bits, S_b >= 0) and the exponent histogram of the
// candidates 1..N-3 are complete in global memory.  The selected set is a
// bitmap; radix select: the exponent digit from the histogram, then 8/8/7
// mantissa bits over the keys still in play (compacted into a list when they
// fit it); keys equal in all bits go to the lower block index.  Writes the
// ascending selection (padded with -1) and its size.
__device__ __forceinline__ void select_unit(const LayerArgs& a, int u, int s, int h, int N, unsigned char* smraw,
                                            int* misc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const int stride = a.key_stride;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smraw);
  uint32_t* phist = keys + stride + 4;          // [kW][kPrivBins] per warp; later a scratch bitmap
  uint32_t* hsum = phist + kW * kPrivBins;      // [kPrivBins] summed
  uint32_t* lkey = hsum + kPrivBins;
  int* lidx = reinterpret_cast<int*>(lkey + kListMax + 4);       // both padded by 4 sentinels
  unsigned* words = reinterpret_cast<unsigned*>(lidx + kListMax + 4);
  int* wbase = reinterpret_cast<int*>(words + (stride + 31) / 32 + 4);
  int* selrow = a.sel + (int64_t)u * K;
  const int nw = (N + 31) / 32;
  unsigned long long tp = a.trace ? global_ns() : 0ull;
  int pk = 0;

  // a. the exponent histogram (then cleared for the next call), an empty bitmap
  {
    unsigned* gh = a.unit_hist + u * kPrivBins;
    if (tid < kPrivBins) {
      hsum[tid] = __ldcg(gh + tid);
      gh[tid] = 0u;
    }
    for (int w = tid; w < nw; w += kT) words[w] = N <= K ? (w < nw - 1 || (N & 31) == 0 ? ~0u : (1u << (N & 31)) - 1u) : 0u;
  }
  __syncthreads();
  int need = K - 3;
  if (N > K && need > 0) {
    const int cand_lo = 1, cand_hi = N - 3;
    find_digit(hsum, kPrivBins, need, misc, lane, warp);
    const uint32_t E = (uint32_t)misc[0];
    const int cntE = misc[2];
    need -= misc[1];
    const bool take_all = cntE == need;
    const bool to_list = !take_all && cntE <= kListMax;
    // b. one pass over the keys (16-byte loads from global memory, coalesced,
    // eight in flight per thread): exponent above E (or at E when all of it
    // is needed) -> selected; at E -> counted for the list.  Selected keys
    // get bit 31 in the shared copy.
    const uint4* src = reinterpret_cast<const uint4*>(a.skeys + (int64_t)u * stride);
    const int n4 = (N + 3) / 4;
    int myc = 0;
    for (int i0 = tid; i0 < n4; i0 += 8 * kT) {
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + k * kT;
        v[k] = i < n4 ? __ldcg(src + i) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + k * kT;
        if (i >= n4) break;
        uint32_t kk[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int b = 4 * i + j;
          if (b >= cand_lo && b <= cand_hi) {
            const uint32_t ex = kk[j] >> 23;
            if (ex > E || (take_all && ex == E)) {
              kk[j] |= 0x80000000u;
              atomicOr(&words[b >> 5], 1u << (b & 31));
            } else if (ex == E) {
              ++myc;
            }
          }
        }
        reinterpret_cast<uint4*>(keys)[i] = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      }
    }
    if (tid == 0) tp = trace_phase(a, u, pk++, 1, tp);
    int m = 0;
    if (to_list) {
      // c. compact the keys at E into the list: CTA-wide offsets, then a
      // second pass over this thread's own chunks (its own shared writes)
      int total;
      int off = cta_exclusive_scan(myc, reinterpret_cast<int*>(hsum), &total, lane, warp);
      m = total;
      if (tid < 4) {  // sentinels up to a multiple of 4: marked, never in play
        lkey[m + tid] = 0x80000000u;
        lidx[m + tid] = 0x7fffffff;
      }
      for (int i = tid; i < n4; i += kT) {
        const uint4 k4 = reinterpret_cast<const uint4*>(keys)[i];
        const uint32_t kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int b = 4 * i + j;
          if (b >= cand_lo && b <= cand_hi && (kk[j] >> 23) == E) {
            lkey[off] = kk[j];
            lidx[off] = b;
            ++off;
          }
        }
      }
    }
    __syncthreads();
    if (tid == 0) tp = trace_phase(a, u, pk++, 2, tp);
    if (!take_all) {
      // d. the keys in play: ranked directly by (key desc, index asc) once
      // they are few and listed, else resolved by mantissa digits
      const int span = cand_hi - cand_lo + 1;
      bool listed = to_list;
      int inplay = cntE;
      uint32_t pfx = E << 23, pm = 0xff800000u;  // in play: (key & pm) == pfx (bit 31 clear)
      bool fin = false;
      uint32_t* mine = phist + warp * kPrivBins;
      for (int level = 1; level <= 4 && !fin; ++level) {
        if (listed && inplay <= kRankMax) {
          // rank of each key in play among those in play; 16-byte broadcast
          // reads of the list (padded with sentinels to a multiple of 4)
          const int m4 = (m + 3) & ~3;
          for (int e = tid; e < m; e += kT) {
            const uint32_t k0 = lkey[e];
            if ((k0 & pm) != pfx) continue;
            const int i0 = lidx[e];
            int rank = 0;
#pragma unroll 4
            for (int f = 0; f < m4; f += 4) {
              const uint4 kf = *reinterpret_cast<const uint4*>(lkey + f);
              const int4 xf = *reinterpret_cast<const int4*>(lidx + f);
              rank += ((kf.x & pm) == pfx) && (kf.x > k0 || (kf.x == k0 && xf.x < i0));
              rank += ((kf.y & pm) == pfx) && (kf.y > k0 || (kf.y == k0 && xf.y < i0));
              rank += ((kf.z & pm) == pfx) && (kf.z > k0 || (kf.z == k0 && xf.z < i0));
              rank += ((kf.w & pm) == pfx) && (kf.w > k0 || (kf.w == k0 && xf.w < i0));
            }
            if (rank < need) atomicOr(&words[i0 >> 5], 1u << (i0 & 31));
          }
          __syncthreads();
          if (tid == 0) tp = trace_phase(a, u, pk++, 9, tp);
          fin = true;
          break;
        }
        if (level == 4) break;  // equal keys left (not listed): the index decides below
        const int shift = level == 1 ? 15 : (level == 2 ? 7 : 0);
        const int nbins = level == 3 ? 128 : 256;
        const uint32_t dmask = (uint32_t)nbins - 1u;
        const int cnt_src = listed ? m : span;
        for (int i = lane; i < kPrivBins; i += 32) mine[i] = 0u;
        __syncwarp();
        for (int e = tid; e < cnt_src; e += kT) {
          const uint32_t key = listed ? lkey[e] : keys[cand_lo + e];
          if ((key & pm) == pfx) atomicAdd(&mine[(key >> shift) & dmask], 1u);
        }
        __syncthreads();
        if (tid < nbins) {
          uint32_t t = 0;
#pragma unroll
          for (int w = 0; w < kW; ++w) t += phist[w * kPrivBins + tid];
          hsum[tid] = t;
        }
        if (tid == 0) misc[3] = 0;
        __syncthreads();
        find_digit(hsum, nbins, need, misc, lane, warp);
        const uint32_t Dg = (uint32_t)misc[0];
        const int cnt = misc[2];
        need -= misc[1];
        const bool all = cnt == need;
        const bool compact = !listed && !all && cnt <= kListMax;
        for (int e0 = warp * 32; e0 < cnt_src; e0 += kT) {
          const int e = e0 + lane;
          bool keep = false;
          uint32_t key = 0u;
          int b = 0;
          if (e < cnt_src) {
            key = listed ? lkey[e] : keys[cand_lo + e];
            b = listed ? lidx[e] : cand_lo + e;
            if ((key & pm) == pfx) {
              const uint32_t dg = (key >> shift) & dmask;
              if (dg > Dg || (all && dg == Dg)) {
                atomicOr(&words[b >> 5], 1u << (b & 31));
                if (listed)
                  lkey[e] = key | 0x80000000u;
                else
                  keys[b] = key | 0x80000000u;
              } else {
                keep = dg == Dg;
              }
            }
          }
          if (compact) {
            const unsigned bal = __ballot_sync(0xffffffffu, keep);
            if (bal) {
              int p0 = 0;
              if (lane == 0) p0 = atomicAdd(misc + 3, __popc(bal));
              p0 = __shfl_sync(0xffffffffu, p0, 0);
              if (keep) {
                const int p = p0 + __popc(bal & ((1u << lane) - 1u));
                lkey[p] = key;
                lidx[p] = b;
              }
            }
          }
        }
        pfx |= Dg << shift;
        pm |= dmask << shift;
        fin = all;
        inplay = cnt;
        __syncthreads();
        if (tid == 0) {
          tp = trace_phase(a, u, pk++, 10 + level, tp);
          if (a.trace)
            trace_item(a, slot_phase(a) + u * 32 + 16 + (level & 15), 6, u, level, (unsigned long long)cnt,
                       (unsigned long long)(listed ? m : -1));
        }
        if (compact) {
          m = misc[3];
          listed = true;
          if (tid < 4) {
            lkey[m + tid] = 0x80000000u;
            lidx[m + tid] = 0x7fffffff;
          }
          __syncthreads();
        }
      }
      if (!fin) {
        // keys equal in every bit are left: the `need` lowest block indices
        // (a scratch bitmap of them, its prefix counts)
        unsigned* tb = phist;
        const int cnt_src = listed ? m : span;
        for (int w = tid; w < nw; w += kT) tb[w] = 0u;
        __syncthreads();
        for (int e = tid; e < cnt_src; e += kT) {
          const uint32_t key = listed ? lkey[e] : keys[cand_lo + e];
          const int b = listed ? lidx[e] : cand_lo + e;
          if ((key & pm) == pfx) atomicOr(&tb[b >> 5], 1u << (b & 31));
        }
        __syncthreads();
        word_prefix(tb, wbase, nw, lane, warp);
        __syncthreads();
        for (int w = tid; w < nw; w += kT) {
          unsigned word = tb[w], take = 0u;
          int rank = wbase[w];
          while (word && rank < need) {
            const unsigned bit = word & (0u - word);
            take |= bit;
            word ^= bit;
            ++rank;
          }
          if (take) atomicOr(&words[w], take);
        }
        __syncthreads();
      }
    }
  }
  if (N > K && tid == 0) {
    atomicOr(&words[0], 1u);
    atomicOr(&words[(N - 2) >> 5], 1u << ((N - 2) & 31));
    atomicOr(&words[(N - 1) >> 5], 1u << ((N - 1) & 31));
  }
  __syncthreads();
  if (tid == 0) tp = trace_phase(a, u, pk++, 3, tp);
  // e. the ascending list from the bitmap and its prefix counts
  const int total = word_prefix(words, wbase, nw, lane, warp);
  const int want = N < K ? N : K;
  if (warp == 0 && lane == 0) {
    if (total != want) set_error(a.status, kDevInternal, s, h, 50);
    a.unit_nsel[u] = total;
  }
  __syncthreads();
  for (int w = tid; w < nw; w += kT) {
    unsigned word = words[w];
    int pos = wbase[w];
    while (word) {
      const int bit = __ffs(word) - 1;
      if (pos < K) selrow[pos] = 32 * w + bit;
      ++pos;
      word &= word - 1u;
    }
  }
  for (int i = want + tid; i < K; i += kT) selrow[i] = -1;
  if (tid == 0) tp = trace_phase(a, u, pk++, 4, tp);
}

// S item: blocks [512 i, 512 i + 512) of a unit.  LSE_g from the unit's
// scoring records; S_b keys of its blocks; their exponent histogram summed
// into the unit's; the unit's last S item selects.
template <int G, int MODE>
__device__ __forceinline__ void s_item(const LayerArgs& a, int item, unsigned char* smraw, unsigned long long t_start) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int s = 0;
  while (s + 1 < a.B && a.ns_first[s + 1] <= item) ++s;
  const int nper = (a.nchunk[s] + 7) / 8;
  const int local = item - a.ns_first[s];
  const int h = local / nper, ci = local % nper;
  const int u = s * a.Hkv + h;
  float* fch = reinterpret_cast<float*>(smraw) + ((sel_region_words(a.key_stride) + 3) & ~3);  // [8][G]
  uint32_t* hist = reinterpret_cast<uint32_t*>(fch + 8 * G);
  int* misc = reinterpret_cast<int*>(hist + kPrivBins);
  for (int i = tid; i < kPrivBins; i += kT) hist[i] = 0u;
  pdl_wait();
  pdl_trigger();
  const unsigned long long t_wait = a.trace ? global_ns() : 0ull;
  bool fits;
  const int L = unit_tokens(a, s, APPEND, &fits);
  const int N = ceil_blocks(L);
  const int b0 = ci * kChunkS;
  const int nb = b0 < N ? min(kChunkS, N - b0) : 0;
  if (nb == 0) {
    if (ci == 0) {  // empty sequence: nothing selected
      for (int i = tid; i < a.K; i += kT) a.sel[(int64_t)u * a.K + i] = -1;
      if (tid == 0) a.unit_nsel[u] = 0;
    }
    return;
  }
  // 1. the u values of the item's blocks (two per thread), in flight while
  // each query head's warp g forms LSE_g from the unit's records (eight per
  // lane in flight) and the item's factors e^(max a - LSE_g)
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = chunk_record(a, s, h, 0);
  float uu[2][G];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int blk = tid + kT * k;
    const int b = b0 + blk;
    const int rec = rec0 + b / kChunk;
#pragma unroll
    for (int g = 0; g < G; ++g)
      uu[k][g] = blk < nb ? __ldcg(a.chunk_u + ((int64_t)rec * G + g) * kChunk + (b % kChunk)) : 0.f;
  }
  if (warp < G) {
    const int g = warp;
    const int cs0 = b0 / kChunk;
    float M = -INFINITY, S = 0.f, fx = 0.f;
    int fj = -1;
    for (int c0 = 0; c0 < nch; c0 += 256) {
      float2 rv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + lane + 32 * k;
        rv[k] = c < nch ? __ldcg(reinterpret_cast<const float2*>(a.chunk_rec + ((int64_t)(rec0 + c) * G + g) * 4))
                        : make_float2(-INFINITY, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + lane + 32 * k;
        if (c >= cs0 && c < cs0 + 8 && c < nch) {
          fx = rv[k].x;
          fj = c - cs0;
        }
        if (rv[k].x != -INFINITY) {
          const float mn = fmaxf(M, rv[k].x);
          S = (M == -INFINITY ? 0.f : S * expf(M - mn)) + rv[k].y * expf(rv[k].x - mn);
          M = mn;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float Mn = fmaxf(M, M2);
      if (Mn != -INFINITY) {
        S = (M == -INFINITY ? 0.f : S * expf(M - Mn)) + (M2 == -INFINITY ? 0.f : S2 * expf(M2 - Mn));
        M = Mn;
      }
    }
    const float lg = M + logf(S);
    if (fj >= 0) fch[fj * G + g] = expf(fx - lg);
  }
  __syncthreads();
  // 2. S_b = sum_g u_{g,b} e^(max a - LSE_g) = sum_g phat sigma2 as keys
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int blk = tid + kT * k;
    if (blk >= nb) continue;
    const int b = b0 + blk;
    const int cl = blk / kChunk;
    float S = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) S = fmaf(uu[k][g], fch[cl * G + g], S);
    S = fmaxf(S, 0.f);
    const uint32_t key = __float_as_uint(S);
    a.skeys[(int64_t)u * a.key_stride + b] = key;
    if (a.scores) a.scores[(int64_t)u * a.score_stride + b] = S;
    if (b >= 1 && b <= N - 3) atomicAdd(&hist[key >> 23], 1u);
  }
  __syncthreads();
  // 3. the item's histogram into the unit's; the unit's last S item selects
  if (tid < kPrivBins && hist[tid]) atomicAdd(a.unit_hist + u * kPrivBins + tid, hist[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int items = (N + kChunkS - 1) / kChunkS;
    const int prev = atomicAdd(a.s2count + u, 1);
    misc[31] = prev == items - 1;
    if (prev == items - 1) a.s2count[u] = 0;
  }
  __syncthreads();
  if (misc[31]) {
    __threadfence();
    const unsigned long long t_sel = a.trace ? global_ns() : 0ull;
    select_unit(a, u, s, h, N, smraw, misc);
    if (tid == 0) trace_item(a, slot_select(a) + u, 3, u, item, t_sel, t_sel);
  }
  if (tid == 0) trace_item(a, slot_items(a) + blockIdx.x, 7, u, ci, t_start, t_wait);
}

// Compensation item: blocks [128 i, 128 i + 128) of a unit.  M_g =
// max_b (ln|b| + zbar) from the unit's scoring records; sum_b w_b vbar_b and
// sum_b w_b, w_b = e^(ln|b| + zbar_b - M_g), summed into the unit's
// accumulator.  The vbar rows are bulk-copied before the wait for the scoring
// kernel (they are final, except the newest block's row, which the scoring
// kernel rewrites and which is read after the wait).
template <int D, int G, int MODE>
__device__ __forceinline__ void comp_item(const LayerArgs& a, int item, unsigned char* smraw, unsigned long long t_start) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr int V = D / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int s = 0;
  while (s + 1 < a.B && a.n2_first[s + 1] <= item) ++s;
  const int local = item - a.n2_first[s];
  const int h = local / a.nchunk2[s], c2 = local % a.nchunk2[s];
  const int u = s * a.Hkv + h;
  bool fits;
  const int L = unit_tokens(a, s, APPEND, &fits);  // seq_len is written by the last kernel only
  const int N = ceil_blocks(L);
  const int b0 = c2 * kChunk2;
  const int nb = b0 < N ? min(kChunk2, N - b0) : 0;
  const bool newest = APPEND && fits && nb > 0 && b0 + nb == N;
  const int nt = nb - (newest ? 1 : 0);
  float* sv = reinterpret_cast<float*>(smraw);
  float* ws = sv + kChunk2 * D;
  float* mref = ws + G * kChunk2;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smraw + comp_bar_offset(D, G));
  const int64_t row0 = row_of(a, s, h, b0);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, nt > 0 ? (uint32_t)nt * D * 4u : 0u);
    if (nt > 0) bulk_g2s(sv, a.vbar + row0 * D, (uint32_t)nt * D * 4u, bar);
  }
  pdl_wait();
  pdl_trigger();
  const unsigned long long t_wait = a.trace ? global_ns() : 0ull;
  if (nb == 0) {
    __syncthreads();
    mbar_wait_bounded(bar, 0, a.status, s, h, 12);
    return;
  }
  // zbar of the item's blocks (in flight while M_g is formed from the records, eight per lane in flight)
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = chunk_record(a, s, h, 0);
  constexpr int NZ = (G * kChunk2 + kT - 1) / kT;
  float zv[NZ];
#pragma unroll
  for (int k = 0; k < NZ; ++k) {
    const int i = tid + kT * k;
    const int g = i / kChunk2, blk = i % kChunk2;
    const int b = b0 + blk;
    zv[k] = (i < G * kChunk2 && blk < nb)
                ? __ldcg(a.chunk_z + ((int64_t)(rec0 + b / kChunk) * G + g) * kChunk + (b % kChunk))
                : 0.f;
  }
  if (warp < G) {
    float m = -INFINITY;
    for (int c0 = 0; c0 < nch; c0 += 256) {
      float mv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + lane + 32 * k;
        mv[k] = c < nch ? __ldcg(a.chunk_rec + ((int64_t)(rec0 + c) * G + warp) * 4 + 2) : -INFINITY;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, mv[k]);
    }
    m = warp_max(m);
    if (lane == 0) {
      mref[warp] = m;
      if (c2 == 0) a.unit_ref[u * G + warp] = m;
    }
  }
  if (newest)
    for (int i = tid; i < D; i += kT) sv[(nb - 1) * D + i] = __ldcg(a.vbar + (row0 + nb - 1) * D + i);
  __syncthreads();
#pragma unroll
  for (int k = 0; k < NZ; ++k) {
    const int i = tid + kT * k;
    if (i >= G * kChunk2) break;
    const int g = i / kChunk2, blk = i % kChunk2;
    float w = 0.f;
    if (blk < nb) {
      const int b = b0 + blk;
      const int n = (b == N - 1) ? L - kBlock * b : kBlock;
      w = expf(ln_n(n) + zv[k] - mref[g]);
    }
    ws[i] = w;
  }
  mbar_wait_bounded(bar, 0, a.status, s, h, 11);
  __syncthreads();
  float acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  for (int blk = warp; blk < nb; blk += kW) {
    float vv[V];
    if (V == 4) {
      const float4 x = *reinterpret_cast<const float4*>(sv + blk * D + lane * 4);
      vv[0] = x.x; vv[1] = x.y; vv[2 % V] = x.z; vv[3 % V] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(sv + blk * D + lane * 2);
      vv[0] = x.x; vv[1 % V] = x.y;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float w = ws[g * kChunk2 + blk];
#pragma unroll
      for (int i = 0; i < V; ++i) acc[g][i] = fmaf(w, vv[i], acc[g][i]);
    }
  }
  __syncthreads();
  float* red = sv;  // [kW][G][D]
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) red[(warp * G + g) * D + lane * V + i] = acc[g][i];
  __syncthreads();
  float* ua = a.unit_acc + (int64_t)u * G * (D + 4);
  for (int i = tid; i < G * D; i += kT) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kW; ++w) t += red[w * G * D + i];
    atomicAdd(ua + (i / D) * (D + 4) + (i % D), t);
  }
  if (warp < G) {
    float t = 0.f;
    for (int blk = lane; blk < kChunk2; blk += 32) t += ws[warp * kChunk2 + blk];
    t = warp_sum(t);
    if (lane == 0) atomicAdd(ua + warp * (D + 4) + D, t);
  }
  if (tid == 0) trace_item(a, slot_items(a) + blockIdx.x, 2, u, c2, t_start, t_wait);
}

// The S items come first in the grid so that they are scheduled first.
template <int D, int G, int MODE>
__global__ void __launch_bounds__(kT) k_select_comp(LayerArgs a) {
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  extern __shared__ __align__(128) unsigned char smraw[];
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  const int ns = SEL ? a.ns_items : 0;
  if ((int)blockIdx.x < ns) {
    if (SEL) s_item<G, MODE>(a, blockIdx.x, smraw, t_start);
  } else if (COMP) {
    comp_item<D, G, MODE>(a, blockIdx.x - ns, smraw, t_start);
  }
}

// Sum of NVAL values over the LPB lanes of a lane group (powers of two,
// NVAL <= LPB).  Halving steps at offsets NVAL/2 .. 1 exchange half of the
// values, then offsets NVAL .. LPB/2 add; lane j ends with the total of value
// index j % NVAL (returned in `idx`).
template <int NVAL, int LPB>
__device__ __forceinline__ float transpose_reduce_lanes(float (&v)[NVAL], int j, int& idx) {
  idx = 0;
#pragma unroll
  for (int c = NVAL; c > 1; c >>= 1) {
    const int off = c / 2;
    const bool up = (j & off) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = up ? v[i] : v[i + c / 2];
      const float keep = up ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    if (up) idx += c / 2;
  }
#pragma unroll
  for (int off = NVAL; off < LPB; off <<= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  return v[0];
}

// ================================================================== 3. attend
// Sum of P values across the warp: lane l ends with the total of value index l % P
// (lanes l and l + P agree when P = 16).
template <int P>
__device__ __forceinline__ float transpose_reduce_warp(float (&v)[P], int lane) {
  int idx;
  return transpose_reduce_lanes<P, 32>(v, lane, idx);
}

constexpr int kAttendWarps = kAttendBlocks;  // selected blocks per attention CTA (one per warp)
static_assert(kAttendWarps == kW, "one selected block per warp of an attention CTA");

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kT) k_attend(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool EXTERNAL = (MODE & kFSelect) == 0;  // selection given by the caller
  constexpr int V = D / 32;
  constexpr int TG = G >= 8 ? 2 : ((32 / G) > 16 ? 16 : (32 / G));  // tokens per reduction group
  constexpr int P = TG * G;                                          // 16 or 32 values per group
  constexpr int W = V / 2;                                           // 32-bit words per token slice
  constexpr int NG = kBlock / TG;
  __shared__ float red_m[kW][G], red_l[kW][G];
  __shared__ __align__(16) float red_a[kW][G][D];
  __shared__ int sh_cnt, sh_bad, sh_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  const int u = blockIdx.x / a.splits, p = blockIdx.x % a.splits;
  const int s = u / a.Hkv, h = u % a.Hkv;
  const int K = a.K;
  float qr[G][V];
  const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) qr[g][i] = qg[g * D + lane * V + i] * InvSqrt<D>::v;
  if (tid == 0) {
    sh_cnt = 0;
    sh_bad = 0;
  }
  pdl_wait();
  const unsigned long long t_wait = a.trace ? global_ns() : 0ull;
  const int L = a.lnew[s], N = ceil_blocks(L);
  const int* selrow = a.sel + (int64_t)u * K;
  __syncthreads();
  int nsel;
  if (EXTERNAL) {
    int cnt = 0, bad = 0;
    for (int i = tid; i < K; i += kT) {
      const int e = __ldcg(selrow + i);
      const int prev = i > 0 ? __ldcg(selrow + i - 1) : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      cnt += ok;
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cnt) atomicAdd(&sh_cnt, cnt);
      if (bad) sh_bad = 1;
    }
    __syncthreads();
    nsel = sh_cnt;
    if (sh_bad && p == 0 && tid == 0) set_error(a.status, kDevBadSelection, s, h, 61);
  } else {
    nsel = __ldcg(a.unit_nsel + u);
  }
  const bool comp = nsel < N;
  float m[G], l[G], acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  }
  const int my_i = p * kAttendWarps + warp;
  int b = -1;
  if (my_i < K) {
    const int e = __ldcg(selrow + my_i);
    const int prev = my_i > 0 ? __ldcg(selrow + my_i - 1) : -1;
    if (e >= 0 && e < N && (my_i == 0 || (prev >= 0 && prev < e))) b = e;
  }
  if (b >= 0) {
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    const int64_t row = row_of(a, s, h, b);
    const unsigned* kp = reinterpret_cast<const unsigned*>(a.k + row * kBlock * D + lane * V);
    const unsigned* vp = reinterpret_cast<const unsigned*>(a.v + row * kBlock * D + lane * V);
    // every load of the block up front: keys, values, its mean value and zbar
    unsigned raw[kBlock][W], rawv[kBlock][W];
#pragma unroll
    for (int j = 0; j < kBlock; ++j) {
      if (W == 2) {
        const uint2 w2 = __ldcg(reinterpret_cast<const uint2*>(kp + j * (D / 2)));
        raw[j][0] = w2.x;
        raw[j][W - 1] = w2.y;
        const uint2 x2 = __ldcg(reinterpret_cast<const uint2*>(vp + j * (D / 2)));
        rawv[j][0] = x2.x;
        rawv[j][W - 1] = x2.y;
      } else {
        raw[j][0] = __ldcg(kp + j * (D / 2));
        rawv[j][0] = __ldcg(vp + j * (D / 2));
      }
    }
    const int rec = chunk_record(a, s, h, b / kChunk);
    float vb[V];
#pragma unroll
    for (int i = 0; i < V; ++i) vb[i] = __ldcg(a.vbar + row * D + lane * V + i);
    const float zb_lane = lane < G ? __ldcg(a.chunk_z + ((int64_t)rec * G + lane) * kChunk + (b % kChunk)) : 0.f;
    float zl[NG];
    const int idx = lane & (P - 1);
    const int jj = idx / G, gl = idx % G;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      float part[P];
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        float kf[V];
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[gi * TG + t][w]));
          kf[2 * w] = x.x;
          kf[2 * w + 1] = x.y;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float acc_t = 0.f;
#pragma unroll
          for (int i = 0; i < V; ++i) acc_t = fmaf(qr[g][i], kf[i], acc_t);
          part[t * G + g] = acc_t;
        }
      }
      zl[gi] = transpose_reduce_warp<P>(part, lane);
    }
    float zmax = -INFINITY;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi)
      if (gi * TG + jj < n) zmax = fmaxf(zmax, zl[gi]);
#pragma unroll
    for (int o = G; o < P; o <<= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    float pl[NG];
    float psum = 0.f;
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
      pl[gi] = (gi * TG + jj < n) ? expf(zl[gi] - zmax) : 0.f;
      psum += pl[gi];
    }
#pragma unroll
    for (int o = G; o < P; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = __shfl_sync(0xffffffffu, zmax, g);
      l[g] = __shfl_sync(0xffffffffu, psum, g);
    }
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        float vf[V];
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&rawv[gi * TG + t][w]));
          vf[2 * w] = x.x;
          vf[2 * w + 1] = x.y;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = __shfl_sync(0xffffffffu, pl[gi], t * G + g);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[g][i] = fmaf(pg, vf[i], acc[g][i]);
        }
      }
    }
    if (comp) {
      // remove this block's own compensation term, which kernel 2 summed for every block
      const float lnn = ln_n(n);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float e = lnn + __shfl_sync(0xffffffffu, zb_lane, g);
        const float mn = fmaxf(m[g], e);
        const float fo = (m[g] == -INFINITY) ? 0.f : expf(m[g] - mn);
        const float fn = expf(e - mn);
        m[g] = mn;
        l[g] = l[g] * fo - fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo - fn * vb[i];
      }
    }
  }
  const unsigned long long t_comp = a.trace ? global_ns() : 0ull;
  // merge the warps into this CTA's partial
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp][g] = m[g];
      red_l[warp][g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < V; ++i) red_a[warp][g][lane * V + i] = acc[g][i];
  }
  __syncthreads();
  float* srec = a.split_rec + ((int64_t)u * a.splits + p) * G * (4 + D);
  for (int i4 = tid; i4 < G * D / 4; i4 += kT) {
    const int g = (4 * i4) / D, col = (4 * i4) % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kW; ++w) M = fmaxf(M, red_m[w][g]);
    float ls = 0.f;
    float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        const float mw = red_m[w][g];
        const float f = (mw == -INFINITY) ? 0.f : expf(mw - M);
        ls += red_l[w][g] * f;
        const float4 x = *reinterpret_cast<const float4*>(&red_a[w][g][col]);
        as.x += x.x * f;
        as.y += x.y * f;
        as.z += x.z * f;
        as.w += x.w * f;
      }
    }
    if (col == 0) {
      srec[g * (4 + D)] = M;
      srec[g * (4 + D) + 1] = ls;
    }
    *reinterpret_cast<float4*>(srec + g * (4 + D) + 4 + col) = as;
  }
  const unsigned long long t_rec = a.trace ? global_ns() : 0ull;
  // the last CTA of the unit merges all partials with the compensation sum
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.mcount + u, 1);
    sh_last = prev == a.splits - 1;
    if (sh_last) a.mcount[u] = 0;
    if (APPEND && blockIdx.x == 0)
      for (int ss = 0; ss < a.B; ++ss) {
        const int Lold = a.seq_len[ss];
        if (Lold >= 0 && Lold < a.cap_blocks[ss] * kBlock)
          a.seq_len[ss] = Lold + 1;
        else
          set_error(a.status, kDevCapacity, ss, -1, 42);
      }
  }
  __syncthreads();
  if (sh_last) {
    __threadfence();
    const float* recs = a.split_rec + (int64_t)u * a.splits * G * (4 + D);
    const float* ua = a.unit_acc + (int64_t)u * G * (D + 4);
    float* out = a.out + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
    const int rs = G * (4 + D);
    for (int i4 = tid; i4 < G * D / 4; i4 += kT) {
      const int g = (4 * i4) / D, col = (4 * i4) % D;
      float M = -INFINITY, ls = 0.f;
      float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q0 = 0; q0 < a.splits; q0 += 8) {
        float mv[8], lv[8];
        float4 av[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int pp = q0 + k;
          if (pp < a.splits) {
            const float* rp = recs + (int64_t)pp * rs + g * (4 + D);
            mv[k] = __ldcg(rp);
            lv[k] = __ldcg(rp + 1);
            av[k] = __ldcg(reinterpret_cast<const float4*>(rp + 4 + col));
          } else {
            mv[k] = -INFINITY;
            lv[k] = 0.f;
            av[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (mv[k] == -INFINITY) continue;
          const float mn = fmaxf(M, mv[k]);
          const float fo = (M == -INFINITY) ? 0.f : expf(M - mn);
          const float fn = expf(mv[k] - mn);
          ls = ls * fo + lv[k] * fn;
          as.x = as.x * fo + av[k].x * fn;
          as.y = as.y * fo + av[k].y * fn;
          as.z = as.z * fo + av[k].z * fn;
          as.w = as.w * fo + av[k].w * fn;
          M = mn;
        }
      }
      if (comp) {
        const float mc = __ldcg(a.unit_ref + u * G + g);
        if (mc != -INFINITY) {
          const float cl = __ldcg(ua + g * (D + 4) + D);
          const float4 ca = __ldcg(reinterpret_cast<const float4*>(ua + g * (D + 4) + col));
          const float mn = fmaxf(M, mc);
          const float fo = (M == -INFINITY) ? 0.f : expf(M - mn);
          const float fn = expf(mc - mn);
          ls = ls * fo + cl * fn;
          as.x = as.x * fo + ca.x * fn;
          as.y = as.y * fo + ca.y * fn;
          as.z = as.z * fo + ca.z * fn;
          as.w = as.w * fo + ca.w * fn;
        }
      }
      const float inv = ls > 0.f ? 1.f / ls : 0.f;
      *reinterpret_cast<float4*>(out + g * D + col) = make_float4(as.x * inv, as.y * inv, as.z * inv, as.w * inv);
    }
  }
  if (tid == 0) trace_item(a, slot_attend(a) + blockIdx.x, sh_last ? 4 : 1, u, p, t_start, t_wait, t_comp, t_rec, 0);
}

// ================================================================== launches
static cudaError_t launch_pdl(const void* fn, dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// raise a kernel's dynamic shared-memory limit once per device and size
static cudaError_t ensure_smem(const void* fn, std::atomic<size_t>* configured, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || configured[dev].load() < bytes) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(bytes);
  }
  return cudaSuccess;
}

template <int D, int G, int MODE>
static cudaError_t launch_chain(const LayerArgs& a_in, cudaStream_t st, int first_pdl) {
  static std::atomic<size_t> cfg1[64], cfg2[64];
  LayerArgs a = a_in;
  void* args[] = {&a};
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr bool ATT = (MODE & kFAttend) != 0;
  cudaError_t e;
  // 1. score: one CTA per 64-block item
  {
    const size_t sm = (size_t)score_smem(D, a.r, G);
    const void* fn = reinterpret_cast<const void*>(&k_score<D, G, MODE>);
    if ((e = ensure_smem(fn, cfg1, sm)) != cudaSuccess) return e;
    if ((e = launch_pdl(fn, dim3(a.total_chunks), sm, st, first_pdl != 0, args)) != cudaSuccess) return e;
  }
  // 2. S items (512 blocks) then compensation items (128 blocks)
  {
    const int grid = (SEL ? a.ns_items : 0) + (COMP ? a.n2_items : 0);
    const size_t sm = (size_t)item_grid_smem(D, G, a.key_stride, SEL, COMP);
    const void* fn = reinterpret_cast<const void*>(&k_select_comp<D, G, MODE>);
    if ((e = ensure_smem(fn, cfg2, sm)) != cudaSuccess) return e;
    if ((e = launch_pdl(fn, dim3(grid), sm, st, true, args)) != cudaSuccess) return e;
  }
  // 3. attention: one CTA per 8 selected blocks
  if (ATT) {
    const void* fn = reinterpret_cast<const void*>(&k_attend<D, G, MODE>);
    if ((e = launch_pdl(fn, dim3(a.B * a.Hkv * a.splits), 0, st, true, args)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, int G>
static cudaError_t launch_chain_dg(const LayerArgs& a, int mode, cudaStream_t st, int first_pdl) {
  switch (mode) {
    case kFusedDecode: return launch_chain<D, G, kFusedDecode>(a, st, first_pdl);
    case kFusedScoreSelect: return launch_chain<D, G, kFusedScoreSelect>(a, st, first_pdl);
    case kFusedAttend: return launch_chain<D, G, kFusedAttend>(a, st, first_pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_chain(const LayerArgs& a, int mode, cudaStream_t st, int first_pdl) {
#define COMPKV_G(DD)                                                 \
  switch (a.G) {                                                     \
    case 1: return launch_chain_dg<DD, 1>(a, mode, st, first_pdl);  \
    case 2: return launch_chain_dg<DD, 2>(a, mode, st, first_pdl);  \
    case 4: return launch_chain_dg<DD, 4>(a, mode, st, first_pdl);  \
    case 8: return launch_chain_dg<DD, 8>(a, mode, st, first_pdl);  \
    default: return cudaErrorInvalidValue;                           \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

size_t chain_smem_bytes(int D, int r, int G, int key_stride) {
  size_t m = (size_t)score_smem(D, r, G);
  if ((size_t)item_grid_smem(D, G, key_stride, true, true) > m) m = (size_t)item_grid_smem(D, G, key_stride, true, true);
  return m;
}

}  // namespace compkv
