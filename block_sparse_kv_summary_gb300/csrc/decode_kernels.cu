// The CompKV decode step (onedev.kr/papers/157) as two kernels chained with
// programmatic dependent launch.
//
// Section "무엇과 다른가" of the CompKV page defines the step per (sequence,
// KV head) "unit": score every 16-token block from its summary, select the
// sink block, the two most recent blocks and the Top-K of S_b, attend exactly
// to the selected blocks and add Mean compensation for the others under one
// normaliser.  Section "어떻게 쓰나" fuses the open block's summary update
// with the K/V pack; here that happens in the first kernel.
//
//   1. k_score  one CTA (two warps) per item of 64 blocks: the item's kbar,
//              vbar and Dbar rows streamed through a 3-stage pipeline of 1-D
//              bulk copies (cp.async.bulk, mbarrier); zbar = q.kbar/sqrt(d),
//              sigma2 = (1/d) sum_t Qsq_t Dbar_t, a = ln|b| + zbar + sigma2/2;
//              per block zbar and sigma2, per query head the item's max a,
//              sum e^(a - max a), max(ln|b| + zbar) and the compensation sums
//              sum_b w vbar_b, w = e^(ln|b| + zbar - that max).  The item
//              holding the newest token appends it first.
//   2. k_post   one thread-block cluster per unit: LSE_g, S_b = sum_g phat
//              sigma2 as order-preserving keys, the forced set and Top-K
//              (a cluster-wide histogram threshold, ties ranked exactly),
//              exact attention over the selected blocks (one per warp) minus
//              their own compensation terms, the compensation sums of every
//              block, and the cluster merge into out = acc / l.
// By Jensen, sum_{j in b} e^{z_j} >= |b| e^{zbar_b}, so removing a selected
// block's mean term never makes a denominator negative.  If every block is
// selected the compensation is skipped (the step is dense attention).
#include <atomic>

#include "compkv_launch.h"

namespace compkv {

constexpr int kT = 256;            // threads of the full radix selection (one CTA)
constexpr int kW = kT / 32;
constexpr int kPrivBins = 256;     // histogram bins of one radix digit
constexpr int kListMax = 2048;     // keys in play compacted into a list once at most this many
constexpr int kRankMax = 512;      // listed keys in play ranked directly once at most this many
constexpr int kDigitShift = 19;      // the histogram digit: key bits 30..19 (exponent, 4 mantissa bits)
constexpr int kHist12 = 1 << (31 - kDigitShift);

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

// Trace slots: scoring CTAs, the CTAs of the units' clusters, then 32 phase
// marks per unit (the full radix selection).
__device__ __forceinline__ int slot_attend(const LayerArgs& a) { return a.total_chunks; }
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
// One warp per scoring item (64 blocks of a unit), one warp per CTA, so that
// nothing in the stream waits on a CTA-wide barrier.  The item's rows arrive
// in groups of kGB blocks through a private kScoreStages-deep pipeline of 1-D
// bulk copies (kbar rows, vbar rows, Dbar rows of the group, one mbarrier per
// stage): while a group is scored the next ones are in flight.
//
// Lane l holds coordinates CPL*l .. CPL*l + CPL-1 (CPL = D/32) of the unit's
// G queries.  A group's zbar partial dots (kGB blocks x G heads per lane) are
// summed across the warp by a halving butterfly: at each xor step a lane keeps
// half of its values and receives its partner's partial of that half, so that
// after five steps lane l holds the full sums of values v = l*VPL .. + VPL-1
// (VPL = max(1, NV/32), NV = kGB*G; for NV < 32, lanes l with the same
// l >> log2(32/NV) hold value v = l >> log2(32/NV)), v = block*G + head.
// sigma2 for r <= 16 is then formed by the lane holding (block, head) from the
// block's Dbar row; for r >= 32 by the same butterfly over the r groups.
//
// Compensation: w_{g,b} = e^(ln|b| + zbar_{g,b} - ref_g) times vbar_b is
// accumulated per lane over its coordinates; ref_g is the running maximum of
// ln|b| + zbar over the blocks seen, and the sums are rescaled when it grows,
// so the item's partial ends relative to mc_g = max_b (ln|b| + zbar).
constexpr int kGB = 8;            // blocks per pipeline group
constexpr int kScoreStages = 3;   // groups in flight per item
constexpr int kScoreWarps = 2;    // warps per item: each takes kGB / kScoreWarps blocks of every group

__host__ __device__ inline int score_stage_floats(int D, int r, bool score, bool comp) {
  return kGB * D + (comp ? kGB * D : 0) + (score ? kGB * ((r + 3) & ~3) : 0);
}
// shared memory: stages | group weights [kGB][G] | Qsq [G][r] | the appended
// block's kbar, vbar, Dbar | mbarriers
__host__ __device__ inline int score_smem(int D, int r, int G, bool score, bool comp) {
  const int rr = (r + 3) & ~3;
  return (kScoreStages * score_stage_floats(D, r, score, comp) + kGB * G + G * rr + 2 * D + rr) * 4 +
         8 * kScoreStages + 16;
}

// A scoring item (64 blocks of a unit) and where its rows are.
struct ScoreChunk {
  int s, h, c, u, L, N, b0, nb, nt, rec;
  bool append;
  int64_t row0;
};

template <bool APPEND>
__device__ __forceinline__ ScoreChunk score_chunk(const LayerArgs& a, int idx) {
  ScoreChunk k;
  k.s = 0;
  while (k.s + 1 < a.B && a.chunk0[k.s + 1] <= idx) ++k.s;
  const int local = idx - a.chunk0[k.s];
  k.h = local / a.nchunk[k.s];
  k.c = local % a.nchunk[k.s];
  k.u = k.s * a.Hkv + k.h;
  bool fits;
  k.L = unit_tokens(a, k.s, APPEND, &fits);
  k.N = ceil_blocks(k.L);
  k.b0 = k.c * kChunk;
  k.nb = k.b0 < k.N ? min(kChunk, k.N - k.b0) : 0;
  k.append = APPEND && fits && k.nb > 0 && k.b0 + k.nb == k.N;
  k.nt = k.nb - (k.append ? 1 : 0);
  k.rec = chunk_record(a, k.s, k.h, k.c);
  k.row0 = row_of(a, k.s, k.h, k.b0);
  return k;
}

// One halving step of the butterfly: N values per lane -> N/2.
template <int N>
__device__ __forceinline__ void halve(float* p, int lane, int o) {
  const bool up = (lane & o) != 0;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float send = up ? p[i] : p[i + N / 2];
    const float keep = up ? p[i + N / 2] : p[i];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
  }
}
// Sum NV per-lane partials across the warp (layout in the section comment).
template <int NV>
__device__ __forceinline__ void butterfly(float (&p)[NV], int lane) {
  if constexpr (NV >= 2) halve<NV>(p, lane, 16); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 16);
  if constexpr (NV >= 4) halve<NV / 2>(p, lane, 8); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 8);
  if constexpr (NV >= 8) halve<NV / 4>(p, lane, 4); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 4);
  if constexpr (NV >= 16) halve<NV / 8>(p, lane, 2); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
  if constexpr (NV >= 32) halve<NV / 16>(p, lane, 1); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
}

template <int CPL>
__device__ __forceinline__ void lds_vec(const float* p, float (&x)[CPL]);
template <>
__device__ __forceinline__ void lds_vec<4>(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
template <>
__device__ __forceinline__ void lds_vec<2>(const float* p, float (&x)[2]) {
  const float2 v = *reinterpret_cast<const float2*>(p);
  x[0] = v.x; x[1] = v.y;
}
template <>
__device__ __forceinline__ void lds_vec<1>(const float* p, float (&x)[1]) { x[0] = *p; }

template <int D, int G, int MODE>
__global__ void __launch_bounds__(32 * kScoreWarps) k_score(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr int CPL = D / 32;                        // coordinates per lane
  constexpr int GBW = kGB / kScoreWarps;              // blocks of a group per warp
  constexpr int NV = GBW * G;                        // (block, head) values of a warp's share of a group
  constexpr int VPL = NV >= 32 ? NV / 32 : 1;        // values a lane ends with
  constexpr int SH = NV >= 32 ? 0 : (NV == 16 ? 1 : (NV == 8 ? 2 : 3));  // log2(32 / NV) for NV < 32
  extern __shared__ __align__(128) float sm[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int r = a.r, rr = (r + 3) & ~3;
  const int stage_f = score_stage_floats(D, r, SCORE, COMP);
  float* sw = sm + kScoreStages * stage_f;   // [kGB][G]
  float* sqs = sw + kGB * G;                 // [G][rr]
  float* pk = sqs + G * rr;                  // appended block: kbar [D], vbar [D], Dbar [rr]
  float* pv = pk + D;
  float* pd = pv + D;
  uint64_t* bars = reinterpret_cast<uint64_t*>(pd + rr);
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  pdl_wait();  // the previous work on the stream may have written this cache
  if (blockIdx.x == 0)
    for (int s = threadIdx.x; s < a.B; s += 32 * kScoreWarps) {
      bool f2;
      a.lnew[s] = unit_tokens(a, s, APPEND, &f2);
    }
  // the item's place in the cache comes from the layout alone: its first
  // copies start before the sequence length (a dependent load) is known; they
  // cover the item's rows up to the capacity (the open block's row is replaced
  // by the append below, rows past the last block are not used)
  int s0 = 0;
  while (s0 + 1 < a.B && a.chunk0[s0 + 1] <= (int)blockIdx.x) ++s0;
  const int loc0 = (int)blockIdx.x - a.chunk0[s0];
  const int h0 = loc0 / a.nchunk[s0], c0 = loc0 % a.nchunk[s0];
  const int cap_nb = min(kChunk, a.cap_blocks[s0] - c0 * kChunk);
  const int64_t row0 = row_of(a, s0, h0, c0 * kChunk);
  const bool dbar_bulk = SCORE && (r & 3) == 0;
  const int ng_cap = (cap_nb + kGB - 1) / kGB;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kScoreStages; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // start the copies of group gi into its stage (rows [8 gi, 8 gi + 8) of the item, up to the capacity)
  const float* gk = a.kbar + row0 * D;
  const float* gv = a.vbar + row0 * D;
  const float* gd = a.dbar + row0 * r;
  auto issue = [=](int gi) {
    if (threadIdx.x != 0) return;
    float* st = sm + (gi % kScoreStages) * stage_f;
    const int rb = gi * kGB, n = max(0, min(kGB, cap_nb - rb));
    const uint32_t bytes = (uint32_t)n * (uint32_t)(D * 4 * (COMP ? 2 : 1) + (dbar_bulk ? r * 4 : 0));
    uint64_t* bar = bars + gi % kScoreStages;
    mbar_arrive_expect_tx(bar, bytes);
    if (n > 0) {
      bulk_g2s(st, gk + rb * D, (uint32_t)n * D * 4u, bar);
      if (COMP) bulk_g2s(st + kGB * D, gv + rb * D, (uint32_t)n * D * 4u, bar);
      if (dbar_bulk) bulk_g2s(st + kGB * D * (COMP ? 2 : 1), gd + rb * r, (uint32_t)n * r * 4u, bar);
    }
  };
  const int pre = min(kScoreStages, ng_cap);
  for (int gi = 0; gi < pre; ++gi) issue(gi);
  const ScoreChunk k = score_chunk<APPEND>(a, blockIdx.x);
  const int ng = (k.nb + kGB - 1) / kGB;
  if (k.nb == 0 || ng <= kScoreStages) pdl_trigger();
  if (k.nb == 0) {
    // nothing to score: let the copies already issued land before the CTA exits
    for (int gi = 0; gi < pre; ++gi) mbar_wait_bounded(bars + gi, 0u, a.status, k.s, k.h, 11);
    return;
  }

  // this lane's coordinates of the G queries
  const float* qbase = a.q + ((int64_t)k.s * a.Hkv * G + (int64_t)k.h * G) * D;
  float q[G][CPL];
#pragma unroll
  for (int g = 0; g < G; ++g) lds_vec<CPL>(qbase + g * D + CPL * lane, q[g]);  // generic load (global)
  // Qsq_{g,t} = sum of q_g^2 over coordinate group t = [t*D/r, (t+1)*D/r)
  if (SCORE && wid == 0) {
    const int gs = D / r;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (gs >= CPL) {
        float t = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) t = fmaf(q[g][c], q[g][c], t);
        for (int o = 1; o < gs / CPL; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if ((lane & (gs / CPL - 1)) == 0) sqs[g * rr + (CPL * lane) / gs] = t;
      } else {
        float t = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          t = fmaf(q[g][c], q[g][c], t);
          if ((c + 1) % gs == 0) {
            sqs[g * rr + (CPL * lane + c) / gs] = t;
            t = 0.f;
          }
        }
      }
    }
  }

  // ---- append: the item holding the open block packs the new token and
  // recomputes that block's summary from its tokens (lane = CPL coordinates,
  // every token; two-pass mean and population variance in fp32 from the
  // exact bf16 values)
  const int patched = k.append ? k.nb - 1 : -1;  // item-local block whose rows come from pk, pv, pd
  if (APPEND && k.append && wid == 0) {
    const int n = k.L - kBlock * (k.N - 1);
    const int64_t row = k.row0 + (k.nb - 1);
    const int c0 = CPL * lane;
    const int64_t nw_off = ((int64_t)k.s * a.Hkv + k.h) * D + c0;
    float kx[kBlock][CPL];
    float ksum[CPL], vsum[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) ksum[c] = vsum[c] = 0.f;
#pragma unroll
    for (int j = 0; j < kBlock; ++j) {
      float kf[CPL], vf[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) kf[c] = vf[c] = 0.f;
      if (j < n) {
        const __nv_bfloat16* ks = (j == n - 1) ? a.k_new + nw_off : a.k + (row * kBlock + j) * D + c0;
        const __nv_bfloat16* vs = (j == n - 1) ? a.v_new + nw_off : a.v + (row * kBlock + j) * D + c0;
        load_bf16<CPL>(ks, kf);
        load_bf16<CPL>(vs, vf);
        if (j == n - 1) {
          store_bf16_raw<CPL>(a.k + (row * kBlock + j) * D + c0, a.k_new + nw_off);
          store_bf16_raw<CPL>(a.v + (row * kBlock + j) * D + c0, a.v_new + nw_off);
        }
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        kx[j][c] = kf[c];
        ksum[c] += kf[c];
        vsum[c] += vf[c];
      }
    }
    float var[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const float mk = ksum[c] / (float)n, mv = vsum[c] / (float)n;
      pk[c0 + c] = mk;
      pv[c0 + c] = mv;
      a.kbar[row * D + c0 + c] = mk;
      a.vbar[row * D + c0 + c] = mv;
      float t = 0.f;
#pragma unroll
      for (int j = 0; j < kBlock; ++j) {
        const float dv = j < n ? kx[j][c] - mk : 0.f;
        t = fmaf(dv, dv, t);
      }
      var[c] = t / (float)n;
    }
    // Dbar_t: mean of the variances over coordinate group t = [t*D/r, (t+1)*D/r)
    const int gs = D / r;
    if (gs >= CPL) {
      float t = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) t += var[c];
      for (int o = 1; o < gs / CPL; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      if ((lane & (gs / CPL - 1)) == 0) {
        const float m = t / (float)gs;
        pd[c0 / gs] = m;
        a.dbar[row * r + c0 / gs] = m;
      }
    } else {
      float t = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        t += var[c];
        if ((c + 1) % gs == 0) {
          const float m = t / (float)gs;
          pd[(c0 + c) / gs] = m;
          a.dbar[row * r + (c0 + c) / gs] = m;
          t = 0.f;
        }
      }
    }
  }
  __syncthreads();  // Qsq and the appended block's rows are in place
  // this lane's values after the butterfly: v = block * G + head (block within this warp's share)
  int vb[VPL], vg[VPL];
  const bool primary = NV >= 32 || (lane & ((1 << SH) - 1)) == 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int v = NV >= 32 ? lane * VPL + i : (lane >> SH);
    vb[i] = v / G;
    vg[i] = v % G;
  }
  constexpr int RPL_MAX = 4;  // Dbar coordinates per lane in the butterfly over the r groups (r = 32 .. 128)
  // per lane and value: running max of a and sum of e^(a - max) (the item's
  // logsumexp parts, reduced at the end)
  float lm[VPL], ll[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    lm[i] = -INFINITY;
    ll[i] = 0.f;
  }
  // compensation state: per head the reference, per lane its coordinates' sums and its values' weight sums
  float ref[G], acc[G][CPL], wsl[VPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    ref[g] = -INFINITY;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[g][c] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) wsl[i] = 0.f;

  for (int gi = 0; gi < ng; ++gi) {
    const float* st = sm + (gi % kScoreStages) * stage_f;
    const float* skb = st;
    const float* svb = st + kGB * D;
    const float* sdb = st + kGB * D * (COMP ? 2 : 1);
    float* swr = sw + wid * GBW * G;  // this warp's weights [GBW][G]
    // this warp's blocks of the group: [rb, rb + nbg), stage rows [wb0, wb0 + nbg)
    const int wb0 = wid * GBW;
    const int rb = gi * kGB + wb0, nbg = max(0, min(GBW, k.nb - rb));
    mbar_wait_bounded(bars + gi % kScoreStages, (uint32_t)(gi / kScoreStages) & 1u, a.status, k.s, k.h, 10);
    if (SCORE && !dbar_bulk) {
      for (int i = threadIdx.x; i < min(kGB, k.nt - gi * kGB) * r; i += 32 * kScoreWarps)
        const_cast<float*>(sdb)[i] = a.dbar[(k.row0 + gi * kGB) * r + i];
      __syncthreads();
    }
    skb += wb0 * D;
    svb += wb0 * D;
    sdb += wb0 * r;
    // zbar partial dots
    float p[NV];
#pragma unroll
    for (int b = 0; b < GBW; ++b) {
      float x[CPL];
      const float* rowp = (rb + b == patched) ? pk : skb + b * D;
      lds_vec<CPL>(rowp + CPL * lane, x);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float t = q[g][0] * x[0];
#pragma unroll
        for (int c = 1; c < CPL; ++c) t = fmaf(q[g][c], x[c], t);
        p[b * G + g] = t;
      }
    }
    butterfly<NV>(p, lane);
    float zb[VPL], cv[VPL], sg[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int bl = rb + vb[i];
      const bool ok = vb[i] < nbg;
      zb[i] = p[i] * InvSqrt<D>::v;
      const int bg = k.b0 + bl;
      cv[i] = ok ? ln_n(bg == k.N - 1 ? k.L - kBlock * bg : kBlock) + zb[i] : -INFINITY;
      sg[i] = 0.f;
      if (SCORE && r <= 16 && ok) {
        const float* drow = (bl == patched) ? pd : sdb + vb[i] * r;
        const float* qsr = sqs + vg[i] * rr;
        float t = 0.f;
#pragma unroll
        for (int tt = 0; tt < 16; ++tt)
          if (tt < r) t = fmaf(qsr[tt], drow[tt], t);
        sg[i] = t;
      }
    }
    if (SCORE && r >= 32) {
      const int rpl = r / 32;
      float ps[NV];
#pragma unroll
      for (int b = 0; b < GBW; ++b) {
        const float* drow = (rb + b == patched) ? pd : sdb + b * r;
        float x[RPL_MAX];
#pragma unroll
        for (int t = 0; t < RPL_MAX; ++t) x[t] = t < rpl ? drow[rpl * lane + t] : 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float t = 0.f;
#pragma unroll
          for (int c = 0; c < RPL_MAX; ++c)
            if (c < rpl) t = fmaf(sqs[g * rr + rpl * lane + c], x[c], t);
          ps[b * G + g] = t;
        }
      }
      butterfly<NV>(ps, lane);
#pragma unroll
      for (int i = 0; i < VPL; ++i) sg[i] = ps[i];
    }
    // zbar and sigma2 per (head, block) to the item's records; a = ln|b| + zbar + sigma2 / 2 into the running parts
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const float s2 = sg[i] / (float)D;
      if (primary && vb[i] < nbg) {
        const int64_t o = ((int64_t)k.rec * G + vg[i]) * kChunk + rb + vb[i];
        a.chunk_z[o] = zb[i];
        if (SCORE) a.chunk_s[o] = s2;
      }
      if (SCORE && primary && vb[i] < nbg) {
        const float av = cv[i] + 0.5f * s2;
        const float mn = fmaxf(lm[i], av);
        ll[i] = (lm[i] == -INFINITY ? 0.f : ll[i] * __expf(lm[i] - mn)) + __expf(av - mn);
        lm[i] = mn;
      }
    }
    if (COMP) {
      // the group's maximum of ln|b| + zbar per head (lanes holding the same head)
      float gm[VPL];
#pragma unroll
      for (int i = 0; i < VPL; ++i) gm[i] = cv[i];
      constexpr int GL = NV >= 32 ? 0 : SH;                                // lowest lane bit of the head
      constexpr int GB2 = (G / VPL) == 1 ? 0 : ((G / VPL) == 2 ? 1 : ((G / VPL) == 4 ? 2 : 3));  // head bits
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const bool head_bit = o >= (1 << GL) && o < (1 << (GL + GB2));
        if (!head_bit)
#pragma unroll
          for (int i = 0; i < VPL; ++i) gm[i] = fmaxf(gm[i], __shfl_xor_sync(0xffffffffu, gm[i], o));
      }
      // every lane learns every head's group maximum and raises its references
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int src = NV >= 32 ? g / VPL : (g << SH);
        float m = gm[0];
#pragma unroll
        for (int i = 1; i < VPL; ++i)
          if (g % VPL == i) m = gm[i];
        m = __shfl_sync(0xffffffffu, m, src);
        if (m > ref[g]) {  // warp-uniform
          const float f = ref[g] == -INFINITY ? 0.f : __expf(ref[g] - m);
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[g][c] *= f;
#pragma unroll
          for (int i = 0; i < VPL; ++i)
            if (vg[i] == g) wsl[i] *= f;
          ref[g] = m;
        }
      }
      // weights of the group's blocks
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        float rg = ref[0];
#pragma unroll
        for (int g = 1; g < G; ++g)
          if (vg[i] == g) rg = ref[g];
        const float w = vb[i] < nbg ? __expf(cv[i] - rg) : 0.f;
        if (primary) {
          swr[vb[i] * G + vg[i]] = w;
          wsl[i] += w;
        }
      }
      __syncwarp();
      for (int b = 0; b < nbg; ++b) {
        float x[CPL], w[G];
        const float* rowp = (rb + b == patched) ? pv : svb + b * D;
        lds_vec<CPL>(rowp + CPL * lane, x);
#pragma unroll
        for (int g0 = 0; g0 < G; g0 += (G >= 4 ? 4 : G)) {
          if constexpr (G >= 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(swr + b * G + g0);
            w[g0] = t4.x; w[g0 + 1] = t4.y; w[g0 + 2] = t4.z; w[g0 + 3] = t4.w;
          } else if constexpr (G == 2) {
            const float2 t2 = *reinterpret_cast<const float2*>(swr + b * G);
            w[0] = t2.x; w[1] = t2.y;
          } else {
            w[0] = swr[b];
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[g][c] = fmaf(w[g], x[c], acc[g][c]);
      }
    }
    __syncthreads();  // the stage and the weights are free again
    if (gi + kScoreStages < ng) {
      issue(gi + kScoreStages);
      if (gi + kScoreStages == ng - 1) pdl_trigger();
    }
  }
  // copies issued up front for groups past the last block (capacity beyond the length) land before the stages are reused
  for (int gi = ng; gi < pre; ++gi) mbar_wait_bounded(bars + gi, 0u, a.status, k.s, k.h, 11);
  const unsigned long long t_scored = a.trace ? global_ns() : 0ull;
  // ---- the item's records, per head: (max a, sum e^(a - max a), max(ln|b| + zbar)),
  // the running parts reduced over the lanes holding that head
  const int rec = k.rec;
  constexpr int GL = NV >= 32 ? 0 : SH;
  constexpr int GB2 = (G / VPL) == 1 ? 0 : ((G / VPL) == 2 ? 1 : ((G / VPL) == 4 ? 2 : 3));
  if (SCORE) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const bool head_bit = o >= (1 << GL) && o < (1 << (GL + GB2));
      if (!head_bit)
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          const float m2 = __shfl_xor_sync(0xffffffffu, lm[i], o), l2 = __shfl_xor_sync(0xffffffffu, ll[i], o);
          const float mn = fmaxf(lm[i], m2);
          if (mn != -INFINITY) {
            ll[i] = (lm[i] == -INFINITY ? 0.f : ll[i] * __expf(lm[i] - mn)) + (m2 == -INFINITY ? 0.f : l2 * __expf(m2 - mn));
            lm[i] = mn;
          }
        }
    }
  }
  // the warps' parts combined through stage 0 (free now): per head (max a, sum, reference,
  // weight sum) and the compensation sums; warp 0 writes the item's records
  float* xr = sm;                       // [kScoreWarps][G][4]
  float* xa = sm + kScoreWarps * G * 4; // [kScoreWarps][G][D]
  float wt[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) wt[i] = primary ? wsl[i] : 0.f;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (vg[i] == g) t += wt[i];
    if (COMP) t = warp_sum(t);
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (primary && vb[i] == 0 && vg[i] == g)
        *reinterpret_cast<float4*>(xr + (wid * G + g) * 4) = make_float4(lm[i], ll[i], ref[g], t);
    if (COMP && wid > 0)
      for (int c = 0; c < CPL; ++c) xa[(wid * G + g) * D + CPL * lane + c] = acc[g][c];
  }
  __syncthreads();
  if (wid == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float M = -INFINITY, Lsum = 0.f, R = -INFINITY, Wsum = 0.f;
      for (int w = 0; w < kScoreWarps; ++w) {
        const float4 e = *reinterpret_cast<const float4*>(xr + (w * G + g) * 4);
        M = fmaxf(M, e.x);
        R = fmaxf(R, e.z);
      }
      float f[kScoreWarps];
      for (int w = 0; w < kScoreWarps; ++w) {
        const float4 e = *reinterpret_cast<const float4*>(xr + (w * G + g) * 4);
        if (e.x != -INFINITY) Lsum += e.y * __expf(e.x - M);
        f[w] = e.z == -INFINITY ? 0.f : __expf(e.z - R);
        Wsum += e.w * f[w];
      }
      if (lane == 0)
        *reinterpret_cast<float4*>(a.chunk_rec + ((int64_t)rec * G + g) * 4) =
            make_float4(SCORE ? M : -INFINITY, SCORE ? Lsum : 0.f, COMP ? R : -INFINITY, 0.f);
      if (COMP) {
        float* dst = a.comp_part + ((int64_t)rec * G + g) * (D + 4);
        float o[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          o[c] = acc[g][c] * f[0];
          for (int w = 1; w < kScoreWarps; ++w) o[c] = fmaf(xa[(w * G + g) * D + CPL * lane + c], f[w], o[c]);
        }
        if constexpr (CPL == 4)
          *reinterpret_cast<float4*>(dst + 4 * lane) = make_float4(o[0], o[1], o[2], o[3]);
        else
          *reinterpret_cast<float2*>(dst + 2 * lane) = make_float2(o[0], o[1]);
        if (lane == 0) dst[D] = Wsum;
      }
    }
  }
  if (threadIdx.x == 0) trace_item(a, blockIdx.x, 0, k.u, k.c, t_start, t_scored);
}

// ================================================================== selection helpers
// The full radix selection of one unit by one CTA (the rare path when more
// keys share the threshold bin than the cluster's list holds).  Its shared
// memory: keys | per-warp histograms | summed histogram | list keys | list
// indices | bitmap | prefix.
__host__ __device__ inline int sel_region_words(int key_stride) {
  const int words = (key_stride + 31) / 32 + 4;
  return key_stride + 4 + (kW + 1) * kPrivBins + 2 * (kListMax + 4) + 2 * words;
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

// Selection for unit u by one CTA: the unit's keys (S_b as
// order-preserving bits, S_b >= 0) and the 12-bit histogram of the
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

  // a. the exponent histogram (sums of the 12-bit histogram's bins), an empty bitmap
  {
    const uint4* gh = reinterpret_cast<const uint4*>(a.hist12 + (int64_t)u * kHist12);
    if (tid < kPrivBins) {
      uint32_t t = 0;
#pragma unroll
      for (int k = 0; k < (kHist12 / kPrivBins) / 4; ++k) {
        const uint4 v = __ldcg(gh + tid * ((kHist12 / kPrivBins) / 4) + k);
        t += v.x + v.y + v.z + v.w;
      }
      hsum[tid] = t;
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

// Transposed reduction of NVAL per-lane values over the warp: at each step a
// lane keeps half of its values and adds its partner's share of that half;
// lane j ends with the total of value index idx (the bits of j select it).
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

// ================================================================== 2. select + attend
// One cluster of C CTAs per unit (C = a.splits <= 16) takes everything after
// the scoring kernel.  CTA rank p owns the unit's scoring items
// [p cpc, (p + 1) cpc) (cpc = ceil(items / C)) and their blocks:
//   a. LSE_g and M_g = max_b (ln|b| + zbar) from the unit's item records;
//      S_b = sum_g u_{g,b} e^(max a - LSE_g) = sum_g phat sigma2 of its
//      blocks as order-preserving keys, a 12-bit histogram of the candidates'
//      (1 .. N-3) top key bits; its items' compensation partials rescaled to
//      M_g (the CTA's compensation share).
//   b. the histograms summed into rank 0's (shared-memory atomics across the
//      cluster); every CTA finds the threshold bin T where the count of
//      larger candidates reaches K - 3; its candidates above T are selected,
//      those in T are listed at rank 0 and ranked by (S_b desc, index asc)
//      unless the whole bin is needed.  If more than kRankMax share T, rank 0
//      runs the full radix selection over the keys instead.
//   c. per-CTA counts give each CTA its offset in the ascending selection; the
//      CTA writes its part of it, and takes the selected blocks at positions
//      8 (it C + p) + warp from their owners' shared memory.
//   d. exact attention over those blocks (one block per warp and round),
//      minus each block's own compensation term; the CTA's partial joins its
//      compensation share; the cluster merges the partials through
//      distributed shared memory into out = acc / l.
// By Jensen, sum_{j in b} e^{z_j} >= |b| e^{zbar_b}, so removing a selected
// block's mean term never makes a denominator negative.  If every block is
// selected the compensation is skipped (the step is dense attention).
template <int P>
__device__ __forceinline__ float transpose_reduce_warp(float (&v)[P], int lane) {
  int idx;
  return transpose_reduce_lanes<P, 32>(v, lane, idx);
}

// Thread-block cluster helpers (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t peer_smem(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 ld_peer_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 ld_peer_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void st_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_peer_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t atom_peer_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

constexpr int kAT = 256;            // threads of a post CTA
constexpr int kAW = kAT / 32;       // its warps: one selected block each per round
constexpr int kMiscInts = 64;
constexpr int kTieCap = 64;         // tie-list entries per CTA of the cluster (more: the full radix selection)

// Shared memory of the post kernel, in 4-byte words:
//   union: selection (histograms [4096] and [256] | keys of the CTA's blocks [cpc * 64] |
//          bitmap [roundup4(cpc * 2) + 4] | every CTA's tie list: keys, indices [16][kTieCap] + 4 each),
//          the full radix selection's region (rank 0, rare), or the attention
//          (per-warp partials [kAW][G][D], m, l [kAW][G])
//   then: compensation share [G][D + 4] | the C CTAs' selections [C][min(cpc * 64, K)] |
//   picks [npick] | incoming partials [items per rank][C][8] | item factors [cpc][G] |
//   LSE, M [G] x 2 | counts [16] | misc [kMiscInts]
__host__ __device__ inline int post_bitmap_words(int cpc) { return ((cpc * 2 + 3) & ~3) + 4; }
struct PostLayout {
  int u_words, stg, stg_w, comp, own, own_n, pick, mstage, fcp, lse, mref, cnts, misc, bars, total_words;
};
__host__ __device__ inline int attend_smem_words(int D, int G) { return kAW * G * D + 2 * kAW * G + 4; }
__host__ __device__ inline int post_items_per_rank(int D, int G, int C) { return (G * D / 4 + C - 1) / C; }
__host__ __device__ inline PostLayout post_layout(int D, int G, int key_stride, int cpc, int K, int npick, bool sel, int C) {
  PostLayout l;
  const int selw = kHist12 + 256 + cpc * kChunk + post_bitmap_words(cpc) + 2 * (16 * kTieCap + 4);
  const int fallback = ((sel_region_words(key_stride) + 3) & ~3) + kMiscInts;
  // attention: the per-warp partials, then per warp its block's K and V rows (bf16) and z, p [kBlock][G]
  l.stg = (attend_smem_words(D, G) + 3) & ~3;
  l.stg_w = kBlock * D + 2 * kBlock * G;
  int u = l.stg + kAW * l.stg_w;
  if (sel && selw > u) u = selw;
  if (sel && fallback > u) u = fallback;
  l.u_words = (u + 3) & ~3;
  l.comp = l.u_words;
  l.own = l.comp + G * (D + 4);
  l.own_n = ((cpc * kChunk < K ? cpc * kChunk : K) + 3) & ~3;
  l.pick = l.own + C * l.own_n;
  l.mstage = l.pick + ((npick + 3) & ~3);
  l.fcp = l.mstage + post_items_per_rank(D, G, C) * C * 8;
  l.lse = l.fcp + ((cpc * G + 3) & ~3);
  l.mref = l.lse + ((G + 3) & ~3);
  l.cnts = l.mref + ((G + 3) & ~3);
  l.misc = l.cnts + 16;
  l.bars = l.misc + kMiscInts;  // kAW mbarriers (8 bytes each)
  l.total_words = l.bars + 2 * kAW;
  return l;
}
__host__ __device__ inline int post_npick(int K, int C, bool loop) { return loop ? ((K + 8 * C - 1) / (8 * C)) * 8 : 8; }

// misc slots
enum : int { kMT = 0, kMAbove, kMCntT, kMListN, kMTotal, kMNsel, kMBad, kMOff };

template <int D, int G, int MODE, bool LOOP>
__global__ void __launch_bounds__(kAT, (LOOP || G >= 8) ? 1 : 2) k_post(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr bool ATT = (MODE & kFAttend) != 0;
  constexpr int V = D / 32;
  constexpr int TG = G >= 8 ? 2 : ((32 / G) > 16 ? 16 : (32 / G));  // tokens per reduction group
  constexpr int P = TG * G;                                          // 16 or 32 values per group
  constexpr int W = V / 2;                                           // 32-bit words per token slice
  constexpr int NG = kBlock / TG;
  extern __shared__ __align__(16) float psm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  const int C = a.splits;
  const int u = blockIdx.x / C;
  const int p = (int)cluster_rank();
  const int s = u / a.Hkv, h = u % a.Hkv;
  const int K = a.K;
  const int npick = post_npick(K, C, LOOP);
  const PostLayout lay = post_layout(D, G, a.key_stride, a.post_cpc, K, npick, SEL, C);
  // selection phase views
  uint32_t* hist = reinterpret_cast<uint32_t*>(psm);  // [4096] top 12 key bits, then [256] top 8 (the exponent)
  uint32_t* chist = hist + kHist12;
  uint32_t* keys = chist + 256;
  unsigned* words = keys + a.post_cpc * kChunk;
  uint32_t* lkey = words + post_bitmap_words(a.post_cpc);
  int* lidx = reinterpret_cast<int*>(lkey + 16 * kTieCap + 4);
  // attention phase views
  float* red_a = psm;                     // [kAW][G][D]
  float* red_m = red_a + kAW * G * D;     // [kAW][G]
  float* red_l = red_m + kAW * G;         // [kAW][G]
  // persistent
  float* ccomp = psm + lay.comp;          // [G][D + 4]: the CTA's compensation share, weight sum at [D]
  int* selall = reinterpret_cast<int*>(psm + lay.own);  // [C][own_n]: CTA q's selected blocks
  int* own = selall + p * lay.own_n;
  float* mstage = psm + lay.mstage;                      // [items per rank][C][8]: acc (4), m, l
  uint64_t* pbars = reinterpret_cast<uint64_t*>(psm + lay.bars);
  int* pick = reinterpret_cast<int*>(psm + lay.pick);
  float* fcp = psm + lay.fcp;
  float* lse = psm + lay.lse;
  float* mref = psm + lay.mref;
  int* cnts = reinterpret_cast<int*>(psm + lay.cnts);
  int* misc = reinterpret_cast<int*>(psm + lay.misc);

  if (ATT && tid == 0) {
    for (int w = 0; w < kAW; ++w) mbar_init(pbars + w, 1);
    fence_mbar_init();
  }
  float qr[G][V];
  if (ATT) {
    const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < V; ++i) qr[g][i] = qg[g * D + lane * V + i] * InvSqrt<D>::v;
  }
  if (SEL) {
    for (int i = tid; i < (kHist12 + 256) / 4; i += kAT) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < kMiscInts) misc[tid] = 0;
    __syncthreads();
    cluster_arrive();  // rank 0's histogram and list counter are zero before any peer adds to them
  } else if (tid < kMiscInts) {
    misc[tid] = 0;
  }
  pdl_wait();
  const unsigned long long t_wait = a.trace ? global_ns() : 0ull;
  // phase marks of rank 0 (tracing aid): mark k = SM clocks since the previous mark
  unsigned long long tp = clock64();
  auto mark = [&](int k) {
    if (a.trace && p == 0 && tid == 0) {
      const unsigned long long c = clock64();
      trace_item(a, slot_phase(a) + u * 32 + k, 5, u, k, tp, c);
      tp = c;
    }
  };
  const int L = a.lnew[s], N = ceil_blocks(L);
  const int nch = (N + kChunk - 1) / kChunk;
  const int cpc = (nch + C - 1) / C;
  const int c_lo = min(nch, p * cpc), c_hi = min(nch, c_lo + cpc);
  const int b_lo = c_lo * kChunk, b_hi = min(N, c_hi * kChunk);
  const int nown = b_hi - b_lo;
  const int rec0 = chunk_record(a, s, h, 0);
  const bool all_sel = N <= K;
  const bool want_keys = SEL && (!all_sel || a.scores);
  // zbar and sigma2 of this thread's first four blocks (4 tid .. 4 tid + 3, one
  // 16-byte load per head and quantity), in flight during the LSE pass
  float4 zv0[G], sv0[G];
  {
    const int i = 4 * tid, b = b_lo + i;
    const int64_t o = ((int64_t)(rec0 + b / kChunk) * G) * kChunk + (b % kChunk);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const bool ld = want_keys && i < nown;
      zv0[g] = ld ? __ldcg(reinterpret_cast<const float4*>(a.chunk_z + o + g * kChunk)) : make_float4(0.f, 0.f, 0.f, 0.f);
      sv0[g] = ld ? __ldcg(reinterpret_cast<const float4*>(a.chunk_s + o + g * kChunk)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // ---- a. LSE_g, M_g and the factors of this CTA's items (one pass over the
  // records when they fit eight per lane; the items' own records stay in registers)
  if ((SEL || COMP) && warp < G) {
    const int g = warp;
    float M = -INFINITY, S = 0.f, MC = -INFINITY;
    float4 rv[8];
    const int ncap = a.nchunk[s];  // the unit's records (loads issued before the item count is known)
    for (int c0 = 0; c0 < ncap; c0 += 256) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + lane + 32 * k;
        rv[k] = c < ncap ? __ldcg(reinterpret_cast<const float4*>(a.chunk_rec + ((int64_t)(rec0 + c) * G + g) * 4))
                         : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (c0 + lane + 32 * k >= nch) rv[k] = make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      float mloc = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        MC = fmaxf(MC, rv[k].z);
        mloc = fmaxf(mloc, rv[k].x);
      }
      if (SEL && mloc != -INFINITY) {
        float sl = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (rv[k].x != -INFINITY) sl += rv[k].y * __expf(rv[k].x - mloc);
        const float mn = fmaxf(M, mloc);
        S = (M == -INFINITY ? 0.f : S * __expf(M - mn)) + sl * __expf(mloc - mn);
        M = mn;
      }
    }
    MC = warp_max(MC);
    float lg = 0.f;
    if (SEL) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float M2 = __shfl_xor_sync(0xffffffffu, M, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
        const float Mn = fmaxf(M, M2);
        if (Mn != -INFINITY) {
          S = (M == -INFINITY ? 0.f : S * __expf(M - Mn)) + (M2 == -INFINITY ? 0.f : S2 * __expf(M2 - Mn));
          M = Mn;
        }
      }
      lg = M + logf(S);
    }
    if (nch <= 256) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = lane + 32 * k;
        if (c >= c_lo && c < c_hi) {
          if (COMP) fcp[(c - c_lo) * G + g] = expf(rv[k].z - MC);
        }
      }
    } else {
      for (int j = lane; j < c_hi - c_lo; j += 32) {
        const float4 r4 = __ldcg(reinterpret_cast<const float4*>(a.chunk_rec + ((int64_t)(rec0 + c_lo + j) * G + g) * 4));
        if (COMP) fcp[j * G + g] = expf(r4.z - MC);
      }
    }
    if (lane == 0) {
      lse[g] = lg;
      mref[g] = MC;
    }
  }
  __syncthreads();
  mark(1);
  // ---- a. keys of this CTA's blocks and their histogram; the compensation share
  if (want_keys) {
    // S_b = sum_g phat sigma2 = sum_g e^(ln|b| + zbar + sigma2/2 - LSE_g) sigma2, four blocks per thread
    for (int i0 = 4 * tid; i0 < nown; i0 += 4 * kAT) {
      float zv[G][4], sv[G][4];
      const int b0 = b_lo + i0;
      const int64_t o = ((int64_t)(rec0 + b0 / kChunk) * G) * kChunk + (b0 % kChunk);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float4 z4 = i0 == 4 * tid ? zv0[g] : __ldcg(reinterpret_cast<const float4*>(a.chunk_z + o + g * kChunk));
        const float4 s4 = i0 == 4 * tid ? sv0[g] : __ldcg(reinterpret_cast<const float4*>(a.chunk_s + o + g * kChunk));
        zv[g][0] = z4.x; zv[g][1] = z4.y; zv[g][2] = z4.z; zv[g][3] = z4.w;
        sv[g][0] = s4.x; sv[g][1] = s4.y; sv[g][2] = s4.z; sv[g][3] = s4.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = i0 + k, b = b0 + k;
        if (i >= nown) break;
        const float lnn = ln_n(b == N - 1 ? L - kBlock * b : kBlock);
        float S = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) S = fmaf(__expf(lnn + zv[g][k] + 0.5f * sv[g][k] - lse[g]), sv[g][k], S);
        S = fmaxf(S, 0.f);
        const uint32_t key = __float_as_uint(S);
        keys[i] = key;
        if (a.scores) a.scores[(int64_t)u * a.score_stride + b] = S;
        if (!all_sel && b >= 1 && b <= N - 3) {
          atomicAdd(&hist[key >> kDigitShift], 1u);
          atomicAdd(&chist[key >> 23], 1u);
        }
      }
    }
  }
  if (COMP) {
    for (int i = tid; i < G * (D + 4) / 4; i += kAT) {
      const int g = (4 * i) / (D + 4), col = (4 * i) % (D + 4);
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < c_hi - c_lo; j0 += 16) {
        float4 v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          v[j] = j0 + j < c_hi - c_lo
                     ? __ldcg(reinterpret_cast<const float4*>(a.comp_part + ((int64_t)(rec0 + c_lo + j0 + j) * G + g) * (D + 4) + col))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float f = j0 + j < c_hi - c_lo ? fcp[(j0 + j) * G + g] : 0.f;
          t.x = fmaf(f, v[j].x, t.x);
          t.y = fmaf(f, v[j].y, t.y);
          t.z = fmaf(f, v[j].z, t.z);
          t.w = fmaf(f, v[j].w, t.w);
        }
      }
      *reinterpret_cast<float4*>(ccomp + g * (D + 4) + col) = t;
    }
  }
  __syncthreads();
  mark(2);

  // ---- b, c. the selection
  int nsel = 0;
  unsigned long long t_sel = 0ull;
  if (SEL) {
    const int nwo = (nown + 31) / 32;
    cluster_wait();  // rank 0's histogram is zero
    if (!all_sel) {
      // the cluster's histograms: the exponent bins at rank 0, the 16 fine bins
      // of exponent e at rank e C / 256.  A CTA adds its counts of bins held
      // elsewhere (its own are in place; peers add to them meanwhile, so it does
      // not read those here): thread t < 256 takes exponent t
      const int own_r = (tid * C) >> 8;
      if (own_r != p) {
        const uint4* hv = reinterpret_cast<const uint4*>(hist) + 4 * tid;
        const uint32_t hr = peer_smem(hist, (uint32_t)own_r);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = hv[k];
          const uint32_t ad = hr + 64u * tid + 16u * k;
          if (v.x) red_peer_add(ad, v.x);
          if (v.y) red_peer_add(ad + 4u, v.y);
          if (v.z) red_peer_add(ad + 8u, v.z);
          if (v.w) red_peer_add(ad + 12u, v.w);
        }
      }
      if (p != 0) {
        const uint32_t cs = chist[tid];
        if (cs) red_peer_add(peer_smem(chist + tid, 0), cs);
      }
    }
    cluster_sync_all();  // rank 0 holds the unit's histogram
    mark(3);
    const int need0 = K - 3;
    bool take_all = true;
    uint32_t T = 0u;
    int need = 0;
    if (!all_sel && need0 > 0) {
      // the threshold exponent from the top of rank 0's exponent histogram (thread t: exponent 255 - t),
      // then the fine bin inside it from its 16 fine bins
      const int ex = 255 - tid;
      const int loc = (int)ld_peer_u32(peer_smem(chist + ex, 0));
      int total;
      const int before = cta_exclusive_scan(loc, misc + kMOff, &total, lane, warp);
      if (before < need0 && need0 <= before + loc) {
        uint32_t c16[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = ld_peer_u4(peer_smem(hist + 16 * ex + 4 * k, (uint32_t)((ex * C) >> 8)));
          c16[4 * k] = v.x;
          c16[4 * k + 1] = v.y;
          c16[4 * k + 2] = v.z;
          c16[4 * k + 3] = v.w;
        }
        int run = before;
        for (int k = 15; k >= 0; --k) {
          if (run < need0 && need0 <= run + (int)c16[k]) {
            misc[kMT] = 16 * ex + k;
            misc[kMAbove] = run;
            misc[kMCntT] = (int)c16[k];
          }
          run += (int)c16[k];
        }
      }
      __syncthreads();
      mark(4);
      T = (uint32_t)misc[kMT];
      need = need0 - misc[kMAbove];
      take_all = misc[kMCntT] == need;
    }
    // classify this CTA's blocks (bitmap of the selected ones); the threshold
    // bin's candidates, when ranking is needed, into this CTA's list
    for (int w = tid; w < nwo; w += kAT) words[w] = 0u;
    __syncthreads();
    for (int i = tid; i < nown; i += kAT) {
      const int b = b_lo + i;
      bool sel = all_sel || b == 0 || b == N - 2 || b == N - 1;
      if (!sel && need0 > 0) {
        const uint32_t key = keys[i];
        const uint32_t bin = key >> kDigitShift;
        if (bin > T || (bin == T && take_all)) {
          sel = true;
        } else if (bin == T) {
          // into every CTA's copy of this CTA's tie list
          const int slot = atomicAdd(misc + kMListN, 1);
          if (slot < kTieCap)
            for (int q = 0; q < C; ++q) {
              st_peer_u32(peer_smem(lkey + p * kTieCap + slot, (uint32_t)q), key);
              st_peer_u32(peer_smem(lidx + p * kTieCap + slot, (uint32_t)q), (uint32_t)b);
            }
        }
      }
      if (sel) atomicOr(&words[i >> 5], 1u << (i & 31));
    }
    if (!take_all) {
      __syncthreads();
      // this CTA's tie count into every CTA
      int* lsz = misc + 16;  // the C list sizes
      if (tid < C) st_peer_u32(peer_smem(lsz + p, (uint32_t)tid), (uint32_t)misc[kMListN]);
      mark(5);
      cluster_sync_all();  // every CTA holds every tie list
      mark(6);
      int m = 0, mx = 0;
      for (int q = 0; q < C; ++q) {
        m += lsz[q];
        mx = max(mx, lsz[q]);
      }
      if (mx <= kTieCap) {
        // rank this CTA's entries among all: region q holds lsz[q] entries; the
        // unused slots hold sentinels (key 0, largest index) that never rank above a listed key
        for (int e = tid; e < C * kTieCap; e += kAT)
          if (e % kTieCap >= lsz[e / kTieCap]) {
            lkey[e] = 0u;
            lidx[e] = 0x7fffffff;
          }
        __syncthreads();
        mark(21);
        (void)m;
        const int cp = lsz[p];
        for (int e = tid; e < cp; e += kAT) {
          const uint32_t k0 = lkey[p * kTieCap + e];
          const int i0 = lidx[p * kTieCap + e];
          int rank = 0;
          for (int f = 0; f < C * kTieCap; f += 4) {
            if (lsz[f / kTieCap] <= f % kTieCap) {  // the rest of region f / kTieCap is empty
              f = (f / kTieCap) * kTieCap + kTieCap - 4;
              continue;
            }
            const uint4 kf = *reinterpret_cast<const uint4*>(lkey + f);
            const int4 xf = *reinterpret_cast<const int4*>(lidx + f);
            rank += (kf.x > k0 || (kf.x == k0 && xf.x < i0));
            rank += (kf.y > k0 || (kf.y == k0 && xf.y < i0));
            rank += (kf.z > k0 || (kf.z == k0 && xf.z < i0));
            rank += (kf.w > k0 || (kf.w == k0 && xf.w < i0));
          }
          // the sentinels (key 0, largest index) never rank above a listed key
          if (rank < need) atomicOr(&words[(i0 - b_lo) >> 5], 1u << ((i0 - b_lo) & 31));
        }
        __syncthreads();
      } else {
        // more keys share the threshold bin than the lists hold: rank 0 runs the
        // full radix selection over the unit's keys (written to global memory here)
        for (int i = tid; i < nown; i += kAT) a.skeys[(int64_t)u * a.key_stride + b_lo + i] = keys[i];
        for (int i = tid; i < kHist12; i += kAT)
          if ((((i >> 4) * C) >> 8) == p) a.hist12[(int64_t)u * kHist12 + i] = hist[i];
        cluster_sync_all();
        if (p == 0) select_unit(a, u, s, h, N, reinterpret_cast<unsigned char*>(psm), misc + kMiscInts - 8);
        cluster_sync_all();
        for (int w = tid; w < nwo; w += kAT) words[w] = 0u;
        __syncthreads();
        for (int i = tid; i < K; i += kAT) {
          const int b = __ldcg(a.sel + (int64_t)u * K + i);
          if (b >= b_lo && b < b_hi) atomicOr(&words[(b - b_lo) >> 5], 1u << ((b - b_lo) & 31));
        }
        __syncthreads();
      }
    }
    __syncthreads();
    // ascending list of this CTA's selected blocks and its count, into every CTA of the cluster
    if (warp == 0) {
      int loc = 0;
      const int per = (nwo + 31) / 32;
      for (int k = 0; k < per; ++k) {
        const int w = per * lane + k;
        if (w < nwo) loc += __popc(words[w]);
      }
      int incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int run = incl - loc;
      for (int k = 0; k < per; ++k) {
        const int w = per * lane + k;
        if (w < nwo) {
          unsigned word = words[w];
          while (word) {
            const int bit = __ffs(word) - 1;
            if (run < lay.own_n) {
              const int b = b_lo + 32 * w + bit;
              own[run] = b;
              for (int q = 0; q < C; ++q)
                if (q != p) st_peer_u32(peer_smem(own + run, (uint32_t)q), (uint32_t)b);
            }
            ++run;
            word &= word - 1u;
          }
        }
      }
      mark(22);
      const int total_own = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) misc[kMTotal] = total_own;
      if (lane < C) st_peer_u32(peer_smem(cnts + p, (uint32_t)lane), (uint32_t)total_own);
    }
    __syncthreads();
    mark(23);
    if (ATT) {
      // the K/V rows (and mean values) of this CTA's selected blocks on their way to L2
      // while the offsets are exchanged; another CTA of the cluster may attend them
      for (int e = tid; e < misc[kMTotal] && e < lay.own_n; e += kAT) {
        const int64_t row = row_of(a, s, h, own[e]);
        prefetch_l2(a.k + row * kBlock * D, kBlock * D * 2);
        prefetch_l2(a.v + row * kBlock * D, kBlock * D * 2);
        if (COMP) prefetch_l2(a.vbar + row * D, D * 4);
      }
    }
    mark(7);
    cluster_sync_all();  // every CTA holds every count and every list
    mark(8);
    int off = 0, tot = 0;
    for (int q = 0; q < C; ++q) {
      off += q < p ? cnts[q] : 0;
      tot += cnts[q];
    }
    nsel = tot;
    int* selrow = a.sel + (int64_t)u * K;
    const int mine = misc[kMTotal];
    for (int i = tid; i < mine; i += kAT)
      if (off + i < K) selrow[off + i] = own[i];
    if (p == 0) {
      for (int i = tot + tid; i < K; i += kAT) selrow[i] = -1;
      if (tid == 0) {
        a.unit_nsel[u] = tot;
        if (tot != (N < K ? N : K)) set_error(a.status, kDevInternal, s, h, 50);
      }
    }
    if (ATT) {
      // this CTA's blocks: positions 8 (it C + p) + w, from their owners' lists
      for (int e = tid; e < npick; e += kAT) {
        const int q = 8 * ((e / 8) * C + p) + (e % 8);
        int b = -1;
        if (q < tot && q < K) {
          int r = 0, base = 0;
          while (r + 1 < C && base + cnts[r] <= q) base += cnts[r++];
          b = selall[r * lay.own_n + (q - base)];
        }
        pick[e] = b;
      }
    }
    t_sel = a.trace ? global_ns() : 0ull;
    mark(9);
    if (!ATT) return;  // no peer reads this CTA's shared memory any more
    __syncthreads();
  } else {
    // the caller's selection: validated (ascending, inside [0, N)), counted
    const int* selrow = a.sel + (int64_t)u * K;
    int cnt = 0, bad = 0;
    for (int i = tid; i < K; i += kAT) {
      const int e = __ldcg(selrow + i);
      const int prev = i > 0 ? __ldcg(selrow + i - 1) : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      cnt += ok;
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cnt) atomicAdd(misc + kMNsel, cnt);
      if (bad) misc[kMBad] = 1;
    }
    __syncthreads();
    nsel = misc[kMNsel];
    if (misc[kMBad] && p == 0 && tid == 0) set_error(a.status, kDevBadSelection, s, h, 61);
    for (int e = tid; e < npick; e += kAT) {
      const int q = 8 * ((e / 8) * C + p) + (e % 8);
      int b = -1;
      if (q < K) {
        const int v = __ldcg(selrow + q);
        const int prev = q > 0 ? __ldcg(selrow + q - 1) : -1;
        if (v >= 0 && v < N && (q == 0 || (prev >= 0 && prev < v))) b = v;
      }
      pick[e] = b;
    }
    __syncthreads();
    t_sel = a.trace ? global_ns() : 0ull;
  }

  // ---- d. attention over this CTA's blocks
  const bool comp = COMP && nsel < N;
  float m[G], l[G], acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  }
  const int idx = lane & (P - 1);
  const int jj = idx / G, gl = idx % G;
  const int rounds = LOOP ? npick / 8 : 1;
  // this warp's staging: the block's K and V rows (bf16 pairs as words), then z and p [kBlock][G]
  uint32_t* wk = reinterpret_cast<uint32_t*>(psm + lay.stg + warp * lay.stg_w);
  uint32_t* wv = wk + kBlock * D / 2;
  float* wz = reinterpret_cast<float*>(wv + kBlock * D / 2);
  float* wp = wz + kBlock * G;
  uint32_t ph = 0u;
  const int hg = lane % G;  // the head of this lane's softmax entries (lane, lane + 32, ...)
  for (int it = 0; it < rounds; ++it) {
    const int b = pick[8 * it + warp];
    if (b < 0) continue;  // warp-uniform
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    const int64_t row = row_of(a, s, h, b);
    __syncwarp();  // the staging's previous contents are read
    if (lane == 0) {
      mbar_arrive_expect_tx(pbars + warp, 2u * kBlock * D * 2u);
      bulk_g2s(wk, a.k + row * kBlock * D, kBlock * D * 2u, pbars + warp);
      bulk_g2s(wv, a.v + row * kBlock * D, kBlock * D * 2u, pbars + warp);
    }
    const int rec = chunk_record(a, s, h, b / kChunk);
    float vb[V];
#pragma unroll
    for (int i = 0; i < V; ++i) vb[i] = comp ? __ldcg(a.vbar + row * D + lane * V + i) : 0.f;
    const float zb_lane = (comp && lane < G) ? __ldcg(a.chunk_z + ((int64_t)rec * G + lane) * kChunk + (b % kChunk)) : 0.f;
    mbar_wait_bounded(pbars + warp, ph, a.status, s, h, 62);
    ph ^= 1u;
    // z = q . k / sqrt(d) of the block's tokens, TG tokens at a time (lanes hold V coordinates)
#pragma unroll 1
    for (int gi = 0; gi < NG; ++gi) {
      float part[P];
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        const uint32_t* kr = wk + (gi * TG + t) * (D / 2) + lane * W;
        float kf[V];
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(kr + w));
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
      const float z = transpose_reduce_warp<P>(part, lane);
      if (lane < P) wz[(gi * TG + jj) * G + gl] = z;
    }
    __syncwarp();
    // per head: the block's max, the running max and the rescale, p = e^(z - max) and its sum
    constexpr int EPL = (kBlock * G + 31) / 32;  // softmax entries per lane
    float zmax = -INFINITY;
#pragma unroll
    for (int k = 0; k < EPL; ++k) {
      const int e = lane + 32 * k;
      if (e < kBlock * G && e / G < n) zmax = fmaxf(zmax, wz[e]);
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
    float mlane = -INFINITY;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(m[g], __shfl_sync(0xffffffffu, zmax, g));
      const float f = (m[g] == -INFINITY) ? 0.f : __expf(m[g] - mn);
      m[g] = mn;
      l[g] *= f;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[g][i] *= f;
      if (g == hg) mlane = mn;
    }
    float psum = 0.f;
#pragma unroll
    for (int k = 0; k < EPL; ++k) {
      const int e = lane + 32 * k;
      if (e < kBlock * G) {
        const float pe = e / G < n ? __expf(wz[e] - mlane) : 0.f;
        wp[e] = pe;
        psum += pe;
      }
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
#pragma unroll
    for (int g = 0; g < G; ++g) l[g] += __shfl_sync(0xffffffffu, psum, g);
    __syncwarp();
    // acc += p v over the block's tokens
#pragma unroll 2
    for (int t = 0; t < n; ++t) {
      const uint32_t* vr = wv + t * (D / 2) + lane * W;
      float vf[V];
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vr + w));
        vf[2 * w] = x.x;
        vf[2 * w + 1] = x.y;
      }
      float pg[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pg[g] = wp[t * G + g];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = fmaf(pg[g], vf[i], acc[g][i]);
    }
    if (comp) {
      // remove this block's own compensation term, which the compensation shares hold for every block
      const float lnn = ln_n(n);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float e = lnn + __shfl_sync(0xffffffffu, zb_lane, g);
        const float mn = fmaxf(m[g], e);
        const float fo = (m[g] == -INFINITY) ? 0.f : __expf(m[g] - mn);
        const float fn = __expf(e - mn);
        m[g] = mn;
        l[g] = l[g] * fo - fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo - fn * vb[i];
      }
    }
  }
  const unsigned long long t_att = a.trace ? global_ns() : 0ull;
  mark(10);
  // the CTA's partial: its warps and its compensation share combined
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp * G + g] = m[g];
      red_l[warp * G + g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < V; ++i) red_a[(warp * G + g) * D + lane * V + i] = acc[g][i];
  }
  __syncthreads();
  // ... pushed, per float4 column item, to the rank that merges that item:
  // rank r merges items [r ipr, (r + 1) ipr)
  const int items = G * D / 4;
  const int ipr = post_items_per_rank(D, G, C);
  for (int i4 = tid; i4 < items; i4 += kAT) {
    const int g = (4 * i4) / D, col = (4 * i4) % D;
    float M = comp ? mref[g] : -INFINITY;
#pragma unroll
    for (int w = 0; w < kAW; ++w) M = fmaxf(M, red_m[w * G + g]);
    float ls = 0.f;
    float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAW; ++w) {
        const float mw = red_m[w * G + g];
        const float f = (mw == -INFINITY) ? 0.f : __expf(mw - M);
        ls += red_l[w * G + g] * f;
        const float4 x = *reinterpret_cast<const float4*>(red_a + (w * G + g) * D + col);
        as.x += x.x * f;
        as.y += x.y * f;
        as.z += x.z * f;
        as.w += x.w * f;
      }
      if (comp) {
        const float f = __expf(mref[g] - M);
        const float4 x = *reinterpret_cast<const float4*>(ccomp + g * (D + 4) + col);
        ls += ccomp[g * (D + 4) + D] * f;
        as.x += x.x * f;
        as.y += x.y * f;
        as.z += x.z * f;
        as.w += x.w * f;
      }
    }
    const int r = i4 / ipr, il = i4 - r * ipr;
    const uint32_t dst = peer_smem(mstage + (il * C + p) * 8, (uint32_t)r);
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "f"(as.x), "f"(as.y), "f"(as.z), "f"(as.w)
                 : "memory");
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1,%2};" ::"r"(dst + 16u), "f"(M), "f"(ls) : "memory");
  }
  if (APPEND && blockIdx.x == 0 && tid == 0)
    for (int ss = 0; ss < a.B; ++ss) {
      const int Lold = a.seq_len[ss];
      if (Lold >= 0 && Lold < a.cap_blocks[ss] * kBlock)
        a.seq_len[ss] = Lold + 1;
      else
        set_error(a.status, kDevCapacity, ss, -1, 42);
    }
  mark(11);
  cluster_sync_all();  // every partial of this rank's items is here; no CTA touches a peer's memory after this
  mark(12);
  const int i_lo = p * ipr, i_hi = min(items, i_lo + ipr);
  if (tid < i_hi - i_lo) {
    const int i4 = i_lo + tid, g = (4 * i4) / D, col = (4 * i4) % D;
    const float* e0 = mstage + tid * C * 8;
    float M = -INFINITY;
    for (int q = 0; q < C; ++q) M = fmaxf(M, e0[q * 8 + 4]);
    float ls = 0.f;
    float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY)
      for (int q = 0; q < C; ++q) {
        const float* e = e0 + q * 8;
        const float mq = e[4];
        const float f = mq == -INFINITY ? 0.f : __expf(mq - M);
        ls = fmaf(e[5], f, ls);
        as.x = fmaf(e[0], f, as.x);
        as.y = fmaf(e[1], f, as.y);
        as.z = fmaf(e[2], f, as.z);
        as.w = fmaf(e[3], f, as.w);
      }
    const float inv = ls > 0.f ? 1.f / ls : 0.f;
    float* out = a.out + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
    *reinterpret_cast<float4*>(out + g * D + col) = make_float4(as.x * inv, as.y * inv, as.z * inv, as.w * inv);
  }
  mark(13);
  if (tid == 0) trace_item(a, slot_attend(a) + blockIdx.x, p == 0 ? 4 : 1, u, p, t_start, t_wait, t_sel, t_att, 0);
}

// ================================================================== launches
static cudaError_t launch_pdl(const void* fn, dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args,
                              int threads = kT, int cluster = 1) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
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
static cudaError_t launch_chain(const LayerArgs& a_in, cudaStream_t st, int first_pdl, cudaEvent_t* ev) {
  static std::atomic<size_t> cfg1[64], cfg3[64];
  LayerArgs a = a_in;
  void* args[] = {&a};
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr bool ATT = (MODE & kFAttend) != 0;
  cudaError_t e;
  // 1. score: one warp (one CTA) per 64-block item
  {
    constexpr bool SCORE = (MODE & kFScore) != 0;
    const size_t sm = (size_t)score_smem(D, a.r, G, SCORE, COMP);
    const void* fn = reinterpret_cast<const void*>(&k_score<D, G, MODE>);
    if ((e = ensure_smem(fn, cfg1, sm)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return e;
    if ((e = launch_pdl(fn, dim3(a.total_chunks), sm, st, first_pdl != 0, args, 32 * kScoreWarps)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return e;
  }
  // 2. select + attend: a cluster of a.splits CTAs per unit
  {
    static std::atomic<size_t> cfg4[64];
    const bool loop = ATT && a.K > kAttendBlocks * a.splits;  // more than one selected block per warp
    const int npick = post_npick(a.K, a.splits, loop);
    const size_t sm = (size_t)post_layout(D, G, a.key_stride, a.post_cpc, a.K, npick, SEL, a.splits).total_words * 4;
    const void* fn = loop ? reinterpret_cast<const void*>(&k_post<D, G, MODE, true>)
                          : reinterpret_cast<const void*>(&k_post<D, G, MODE, false>);
    if ((e = ensure_smem(fn, loop ? cfg4 : cfg3, sm)) != cudaSuccess) return e;
    if (a.splits > 8 && (e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
      return e;
    if (ev && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return e;
    if ((e = launch_pdl(fn, dim3(a.B * a.Hkv * a.splits), sm, st, true, args, kAT, a.splits)) != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[3], st)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D, int G>
static cudaError_t launch_chain_dg(const LayerArgs& a, int mode, cudaStream_t st, int first_pdl, cudaEvent_t* ev) {
  switch (mode) {
    case kFusedDecode: return launch_chain<D, G, kFusedDecode>(a, st, first_pdl, ev);
    case kFusedScoreSelect: return launch_chain<D, G, kFusedScoreSelect>(a, st, first_pdl, ev);
    case kFusedAttend: return launch_chain<D, G, kFusedAttend>(a, st, first_pdl, ev);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_chain(const LayerArgs& a, int mode, cudaStream_t st, int first_pdl, cudaEvent_t* ev) {
#define COMPKV_G(DD)                                                 \
  switch (a.G) {                                                     \
    case 1: return launch_chain_dg<DD, 1>(a, mode, st, first_pdl, ev);  \
    case 2: return launch_chain_dg<DD, 2>(a, mode, st, first_pdl, ev);  \
    case 4: return launch_chain_dg<DD, 4>(a, mode, st, first_pdl, ev);  \
    case 8: return launch_chain_dg<DD, 8>(a, mode, st, first_pdl, ev);  \
    default: return cudaErrorInvalidValue;                           \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

size_t chain_smem_bytes(int D, int r, int G, int key_stride, int post_cpc, int K, int splits) {
  size_t m = (size_t)score_smem(D, r, G, true, true);
  const bool loop = K > kAttendBlocks * splits;
  const size_t pm =
      (size_t)post_layout(D, G, key_stride, post_cpc, K, post_npick(K, splits, loop), true, splits).total_words * 4;
  return pm > m ? pm : m;
}

}  // namespace compkv
