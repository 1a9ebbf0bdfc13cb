// The summary stream of the CompKV decode step (onedev.kr/papers/157).
//
// Section "무엇과 다른가" scores every 16-token block of a (sequence, KV
// head) "unit" from its summary {|b|, kbar_b, Dbar_b, vbar_b}:
//   zbar_{g,b}   = q_g . kbar_b / sqrt(d)
//   sigma2_{g,b} = (1/d) sum_t (sum_{i in G_t} q_{g,i}^2) (Dbar_b)_t
//   a_{g,b}      = ln|b| + zbar + sigma2 / 2        (log of the mass estimate)
// and Mean compensation ("어떻게 동작하나") needs, over the unselected blocks,
// sum_b |b| e^{zbar_{g,b}} vbar_b and sum_b |b| e^{zbar_{g,b}}.  This kernel
// streams every summary row of the layer once and leaves, per block, zbar and
// sigma2, and per segment of blocks the logsumexp parts of a and the
// compensation sums over all of its blocks (the post kernel removes the
// selected blocks' own terms).  A call that appends leaves the open block
// (the one receiving the new token) to the post kernel, which packs the token
// and recomputes that block's summary ("어떻게 쓰나": the fused update of the
// current block's statistics and the K/V pack).
//
// Grid: P persistent CTAs of kWarps warps.  The layer's units are cut into
// segments (decode_common.cuh); CTA i takes segments i, i + P, ...  Within a
// segment, stage k (SB consecutive blocks: their kbar, vbar and Dbar rows,
// one 1-D bulk copy each) belongs to warp k % kWarps, which owns one
// shared-memory slot and issues its own copies, so no warp waits on another
// while the stream runs.  The kbar and Dbar rows and the vbar rows of a stage
// arrive on two barriers: the next stage's kbar rows are in flight while the
// warp forms this stage's compensation sums, and its vbar rows while it scores
// the next stage.  In a call that appends, the first Q CTAs of the grid
// recompute the units' open blocks instead (one warp per unit).
//
// Per stage a warp forms the SB x G partial dots q_g . kbar_b over its lanes'
// coordinates (lane l holds coordinates CPL*l .. CPL*l + CPL - 1) and sums
// them across the warp with a halving butterfly: at each xor step a lane keeps
// half of its values and receives its partner's partial of that half, so the
// NV = SB*G values end one per lane (or replicated over 32/NV lanes).  With
// long Dbar rows (r = 32 RPL, RPL = 2 or 4) sigma2 takes the same form: each
// lane reads its RPL coordinates of the Qsq and Dbar rows as one vector, and a
// second butterfly sums the partials.  The kernel has an instance that records
// the work-item trace and one without any trace code.
#include "compkv_launch.h"
#include "decode_common.cuh"

namespace compkv {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlots = 1;  // stage slots per warp (two CTAs per multiprocessor)

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

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// floats of one stage slot: kbar rows | vbar rows | Dbar rows (4 floats per row at least)
__host__ __device__ inline int stream_slot_floats(int D, int r, int G, bool score, bool comp) {
  const int sb = stage_blocks(r, G);
  return sb * D + (comp ? sb * D : 0) + (score ? sb * (r < 4 ? 4 : r) : 0);
}
// shared memory: slots | per-warp weights [kWarps][sb][G] | per-warp Qsq [kWarps][G][rr] |
// plan (ints) | mbarriers
__host__ __device__ inline int stream_smem_bytes(int D, int r, int G, bool score, bool comp) {
  const int rr = (r + 3) & ~3;
  const int sb = stage_blocks(r, G);
  const int floats = kWarps * kSlots * stream_slot_floats(D, r, G, score, comp) + kWarps * sb * G +
                     (long_dbar(r) ? 1 : kWarps) * G * rr;
  return floats * 4 + (3 * kMaxBatch + 8) * 4 + 8 * (2 * kWarps * kSlots + 2) + 64;
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
// Sum NV per-lane partials across the warp.  Afterwards lane l holds the
// total of value v = l >> log2(32 / NV) (NV <= 32; lanes with equal v agree).
template <int NV>
__device__ __forceinline__ void butterfly(float (&p)[NV], int lane) {
  static_assert(NV <= 32, "one value per lane at most");
  if constexpr (NV >= 2) halve<NV>(p, lane, 16); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 16);
  if constexpr (NV >= 4) halve<NV / 2>(p, lane, 8); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 8);
  if constexpr (NV >= 8) halve<NV / 4>(p, lane, 4); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 4);
  if constexpr (NV >= 16) halve<NV / 8>(p, lane, 2); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 2);
  if constexpr (NV >= 32) halve<NV / 16>(p, lane, 1); else p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
}

// CPL floats of global memory through L2 only: every global input of these
// kernels may have been written by the kernel before (a chain launched with
// programmatic dependent launch), so no load may be served by a stale L1 line.
template <int CPL>
__device__ __forceinline__ void ldcg_vec(const float* p, float (&x)[CPL]);
template <>
__device__ __forceinline__ void ldcg_vec<4>(const float* p, float (&x)[4]) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
template <>
__device__ __forceinline__ void ldcg_vec<2>(const float* p, float (&x)[2]) {
  const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
  x[0] = v.x; x[1] = v.y;
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

// The open block of unit u (the block this call's token joins), by one warp.  Lane l
// holds the 8-coordinate chunk c = l % CH (CH = D / 8 chunks of a row) of the
// tokens TPL (l / CH) .. TPL (l / CH) + TPL - 1 (TPL = D / 16), loaded as
// 16-byte vectors; sums over the token groups are exchanged by xor shuffles.
// Mean and population variance are two-pass in fp32 from the exact bf16
// values; a_g = ln n + zbar_g + sigma2_g / 2 with
// sigma2_g = (1/d) sum_i q_gi^2 Dbar_t(i) = sum_i qr_gi^2 Dbar_t(i), qr = q / sqrt(d).
// The warp also stores the token and the block's kbar, vbar and Dbar rows,
// and writes a_g to the scratch for the post kernel.  A sequence at capacity
// keeps its cache and is reported (status word, site 1).
template <int D, int G>
__device__ __noinline__ void open_block_warp(const LayerArgs& a, int u, int lane) {
  const int s = u / a.Hkv, h = u % a.Hkv;
  bool fits = false;
  const int L = call_tokens(__ldcg(a.seq_len + s), a.cap_blocks[s], true, &fits);
  if (!fits) {
    if (h == 0 && lane == 0) set_error(a.status, kDevCapacity, s, -1, 1);
    return;
  }
  const int N = ceil_blocks(L);
  const int64_t row0 = row_of(a, s, h, 0);
  const bool owner = true;
  float* anm = a.anm + (int64_t)u * G;

  constexpr int CH = D / 8;
  constexpr int TPL = D / 16;
  const int n = L - kBlock * (N - 1);
  const int64_t row = row0 + (N - 1);
  const int c = lane % CH, tg = lane / CH;
  const int64_t nw = ((int64_t)s * a.Hkv + h) * D;
  const uint4* knew = reinterpret_cast<const uint4*>(a.k_new + nw) + c;
  const uint4* vnew = reinterpret_cast<const uint4*>(a.v_new + nw) + c;
  uint4* kb = reinterpret_cast<uint4*>(a.k + row * kBlock * D) + c;
  uint4* vb = reinterpret_cast<uint4*>(a.v + row * kBlock * D) + c;
  const uint4 kn = __ldcg(knew), vn = __ldcg(vnew);
  if (owner && tg == 0) {
    kb[(n - 1) * CH] = kn;
    vb[(n - 1) * CH] = vn;
  }
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  uint4 kx[TPL], vx[TPL];
#pragma unroll
  for (int i = 0; i < TPL; ++i) {
    const int j = tg * TPL + i;
    kx[i] = j < n - 1 ? __ldcg(kb + j * CH) : (j == n - 1 ? kn : z4);
    vx[i] = !owner ? z4 : (j < n - 1 ? __ldcg(vb + j * CH) : (j == n - 1 ? vn : z4));
  }
  float ks[8], vs[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) ks[e] = vs[e] = 0.f;
#pragma unroll
  for (int i = 0; i < TPL; ++i) {
    const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kx[i]);
    const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&vx[i]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 kf = __bfloat1622float2(k2[e]), vf = __bfloat1622float2(v2[e]);
      ks[2 * e] += kf.x;
      ks[2 * e + 1] += kf.y;
      vs[2 * e] += vf.x;
      vs[2 * e + 1] += vf.y;
    }
  }
#pragma unroll
  for (int o = CH; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ks[e] += __shfl_xor_sync(0xffffffffu, ks[e], o);
      vs[e] += __shfl_xor_sync(0xffffffffu, vs[e], o);
    }
  const float inv = 1.f / (float)n;
  float mk[8], var[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    mk[e] = ks[e] * inv;
    var[e] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < TPL; ++i) {
    if (tg * TPL + i < n) {
      const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kx[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 kf = __bfloat1622float2(k2[e]);
        const float d0 = kf.x - mk[2 * e], d1 = kf.y - mk[2 * e + 1];
        var[2 * e] = fmaf(d0, d0, var[2 * e]);
        var[2 * e + 1] = fmaf(d1, d1, var[2 * e + 1]);
      }
    }
  }
#pragma unroll
  for (int o = CH; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) var[e] += __shfl_xor_sync(0xffffffffu, var[e], o);
  // Dbar_t over coordinate group t = [t*D/r, (t+1)*D/r); dm[e]: the mean of coordinate e's group
  const int r = a.r, gs = D / r;
  float dm[8];
  if (gs >= 8) {
    float t = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) t += var[e] * inv;
#pragma unroll 1
    for (int o = 1; o < gs / 8; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const float m = t / (float)gs;
#pragma unroll
    for (int e = 0; e < 8; ++e) dm[e] = m;
    if (owner && tg == 0 && (c & (gs / 8 - 1)) == 0) a.dbar[row * r + (8 * c) / gs] = m;
  } else {
    // gs = 1, 2 or 4: the groups of the chunk's 8 coordinates, by pairwise sums (gs is a power of two)
#pragma unroll
    for (int e = 0; e < 8; ++e) dm[e] = var[e] * inv;
    if (gs >= 2) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) dm[e] = dm[e + 1] = 0.5f * (dm[e] + dm[e + 1]);
    }
    if (gs >= 4) {
#pragma unroll
      for (int e = 0; e < 8; e += 4) dm[e] = dm[e + 1] = dm[e + 2] = dm[e + 3] = 0.5f * (dm[e] + dm[e + 2]);
    }
    if (owner && tg == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (e % gs == 0) a.dbar[row * r + (8 * c + e) / gs] = dm[e];
    }
  }
  if (owner && tg == 0) {
    float4* kr = reinterpret_cast<float4*>(a.kbar + row * D + 8 * c);
    float4* vr = reinterpret_cast<float4*>(a.vbar + row * D + 8 * c);
    kr[0] = make_float4(mk[0], mk[1], mk[2], mk[3]);
    kr[1] = make_float4(mk[4], mk[5], mk[6], mk[7]);
    vr[0] = make_float4(vs[0] * inv, vs[1] * inv, vs[2] * inv, vs[3] * inv);
    vr[1] = make_float4(vs[4] * inv, vs[5] * inv, vs[6] * inv, vs[7] * inv);
  }
  const float* qg = a.q + ((int64_t)s * a.Hkv + h) * G * D + 8 * c;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float4 q0 = __ldcg(reinterpret_cast<const float4*>(qg + g * D));
    const float4 q1 = __ldcg(reinterpret_cast<const float4*>(qg + g * D + 4));
    const float qr[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float z = 0.f, sg = 0.f;
    if (tg == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = qr[e] * InvSqrt<D>::v;
        z = fmaf(x, mk[e], z);
        sg = fmaf(x * x, dm[e], sg);
      }
    }
    z = warp_sum(z);
    sg = warp_sum(sg);
    if (lane == 0) anm[g] = ln_count(n) + z + ((a.variant & kVarFirstOrderMass) ? 0.f : 0.5f * sg);
  }
}

// TRACE: the work-item trace is recorded (a.trace is set); the instance without it carries no
// trace code.
template <int D, int G, int MODE, int SB, int RPL, bool TRACE>
__global__ void __launch_bounds__(kThreads, 2) k_stream(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr bool SELMODE = (MODE & kFSelect) != 0;
  constexpr bool RB = RPL > 0;                // long Dbar rows: r = 32 RPL coordinates, RPL per lane
  constexpr int CPL = D / 32;
  constexpr int NV = SB * G;                  // (block, head) values of a stage
  constexpr int SH = ilog2(32 / NV);          // lanes per value = 1 << SH
  constexpr int GB = ilog2(G);                // lane bits that select the head
  static_assert(NV <= 32, "stage values exceed the warp");
  extern __shared__ __align__(128) float sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = a.r, rr = (r + 3) & ~3, rs = r < 4 ? 4 : r;
  const int Gp = pad_g(G);
  const int slot_f = stream_slot_floats(D, r, G, SCORE, COMP);
  float* slots = sm;
  float* sw = slots + kWarps * kSlots * slot_f;  // [kWarps][SB][G]
  float* sqs = sw + kWarps * SB * G;             // [kWarps][G][rr] (one copy per warp; shared when RB)
  int* sL = reinterpret_cast<int*>(sqs + (RB ? 1 : kWarps) * G * rr);  // [kMaxBatch] tokens of each sequence in this call
  int* sN = sL + kMaxBatch;                      // [kMaxBatch] blocks streamed
  int* soff = sN + kMaxBatch;                    // [kMaxBatch + 1] first segment of each sequence
  int* sseg = soff + kMaxBatch + 1;
  int* sbad = sseg + 1;                          // a wait of this CTA ran out
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sbad + 1) + 7) & ~uintptr_t(7));
  const unsigned long long t_start = TRACE ? global_ns() : 0ull;
  if (threadIdx.x < 2 * kWarps) mbar_init(bars + threadIdx.x, 1);  // per warp: kbar/Dbar copies, vbar copies
  if (threadIdx.x == 0) {
    *sbad = 0;
    fence_mbar_init();
  }
  // the previous work on the stream may have written this cache and its lengths
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < a.Q) {
    // the open blocks: warp w of CTA c takes the units c * kWarps + w + Q * kWarps * k
    if (APPEND) {
      const int units = a.B * a.Hkv;
#pragma unroll 1
      for (int u = blockIdx.x * kWarps + warp; u < units; u += a.Q * kWarps) open_block_warp<D, G>(a, u, lane);
    }
    if (TRACE && threadIdx.x == 0 && (int)blockIdx.x < a.trace_cap) {
      unsigned long long* rr = a.trace + 1 + 8 * (int64_t)blockIdx.x;
      rr[0] = ((unsigned long long)blockIdx.x << 32);
      rr[1] = 0ull;
      rr[2] = t_start;
      rr[3] = t_start;
      rr[4] = t_start;
      rr[5] = global_ns();
      rr[6] = 0ull;
      rr[7] = 0ull;
    }
    return;
  }
  const int cta = (int)blockIdx.x - a.Q;  // this CTA among the P that stream
  if (warp == 0) {
    const int s0 = lane, s1 = lane + 32;
    bool f0 = false, f1 = false;
    if (s0 < a.B) {
      sL[s0] = call_tokens(__ldcg(a.seq_len + s0), a.cap_blocks[s0], APPEND, &f0);
      sN[s0] = streamed_blocks(sL[s0], APPEND && f0, SELMODE, a.K, a.scores != nullptr);
    }
    if (s1 < a.B) {
      sL[s1] = call_tokens(__ldcg(a.seq_len + s1), a.cap_blocks[s1], APPEND, &f1);
      sN[s1] = streamed_blocks(sL[s1], APPEND && f1, SELMODE, a.K, a.scores != nullptr);
    }
    __syncwarp();
    plan_warp(sN, a.B, a.Hkv, a.P, SB, soff, sseg, lane);
  }
  __syncthreads();
  const int seg = *sseg, total = soff[a.B];
  const unsigned long long t_plan = TRACE ? global_ns() : 0ull;
  unsigned long long t_first = 0ull, t_r1 = 0ull, t_r2 = 0ull, t_r3 = 0ull;
  int nseg_done = 0;
  uint32_t usesK = 0, usesV = 0;  // stages whose kbar/Dbar (vbar) this warp has consumed: the barriers' phases
  float* swr = sw + warp * SB * G;
  float* sqw = RB ? sqs : sqs + warp * G * rr;  // this warp's Qsq [G][rr]
  // this lane's (block, head) value of a stage
  const int vv = lane >> SH, vb = vv / G, vg = vv % G;
  const bool primary = (lane & ((1 << SH) - 1)) == 0;

  for (int si = cta; si < total; si += a.P) {
    int s, h, b0, nb;
    plan_segment(si, a.B, a.Hkv, sN, soff, seg, &s, &h, &b0, &nb);
    const int L = sL[s], N = ceil_blocks(L);  // N: all blocks (the last may be partial)
    const int64_t row0 = row_of(a, s, h, b0);
    const int ns = (nb + SB - 1) / SB;  // stages of the segment
    const bool comp = COMP && !(a.variant & kVarNoCompensation) && (!SELMODE || N > a.K);
    const bool dbulk = SCORE && r >= 4;
    // the summaries are read once per call: evict-first in L2, so that they do not
    // push the kernels' code and the small scratch arrays out of it
    const uint64_t pol = policy_evict_first();
    // ---- this warp's copies: its j-th stage of the segment is stage warp + kWarps j.  The kbar
    // and Dbar rows and the vbar rows of a stage arrive on two barriers, so that the next stage's
    // kbar rows are in flight while this stage's compensation sums are formed, and its vbar rows
    // while the next stage is scored
    float* st = slots + warp * slot_f;
    auto issueK = [&](int k) {
      const int rb = k * SB, n = min(SB, nb - rb);
      uint64_t* bar = bars + 2 * warp;
      mbar_arrive_expect_tx(bar, (uint32_t)n * (uint32_t)(D * 4 + (dbulk ? r * 4 : 0)));
      bulk_g2s_hint(st, a.kbar + (row0 + rb) * D, (uint32_t)n * D * 4u, bar, pol);
      if (dbulk) bulk_g2s_hint(st + SB * D * (comp ? 2 : 1), a.dbar + (row0 + rb) * r, (uint32_t)n * r * 4u, bar, pol);
    };
    auto issueV = [&](int k) {
      const int rb = k * SB, n = min(SB, nb - rb);
      uint64_t* bar = bars + 2 * warp + 1;
      mbar_arrive_expect_tx(bar, (uint32_t)n * D * 4u);
      bulk_g2s_hint(st + SB * D, a.vbar + (row0 + rb) * D, (uint32_t)n * D * 4u, bar, pol);
    };
    const int mine = warp < ns ? (ns - 1 - warp) / kWarps + 1 : 0;  // stages of this warp
    if (lane == 0 && mine > 0) {
      // (the previous segment's record used the slots with ordinary stores)
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issueK(warp);
      if (comp) issueV(warp);
    }
    // ---- queries of the unit: this lane's coordinates, scaled by 1/sqrt(d); Qsq per warp
    // (one shared copy, and a CTA barrier, for long Dbar rows)
    const float* qbase = a.q + ((int64_t)s * a.Hkv + h) * G * D;
    float q[G][CPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      ldcg_vec<CPL>(qbase + g * D + CPL * lane, q[g]);
#pragma unroll
      for (int c = 0; c < CPL; ++c) q[g][c] *= InvSqrt<D>::v;
    }
    if (SCORE && (!RB || warp == 1)) {
      // Qsq_{g,t} = sum of q_g^2 over coordinate group t = [t*D/r, (t+1)*D/r) (q unscaled: x d)
      const int gs = D / r;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (gs >= CPL) {
          float t = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) t = fmaf(q[g][c], q[g][c], t);
          for (int o = 1; o < gs / CPL; o <<= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
          if ((lane & (gs / CPL - 1)) == 0) sqw[g * rr + (CPL * lane) / gs] = t * (float)D;
        } else {
          float t = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            t = fmaf(q[g][c], q[g][c], t);
            if ((c + 1) % gs == 0) {
              sqw[g * rr + (CPL * lane + c) / gs] = t * (float)D;
              t = 0.f;
            }
          }
        }
      }
    }
    if (RB)
      __syncthreads();  // the shared Qsq is in place
    else
      __syncwarp();     // this warp's Qsq is in place

    // ---- stream this warp's stages
    float lm = -INFINITY, ll = 0.f;        // this lane's value: running max of a, sum of e^(a - max)
    float ref[G], acc[G][CPL], wsl = 0.f;  // compensation: per-head reference, numerator, weight sum
#pragma unroll
    for (int g = 0; g < G; ++g) {
      ref[g] = -INFINITY;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[g][c] = 0.f;
    }
    bool bad = false;
    for (int j = 0; j < mine; ++j) {
      const int k = warp + kWarps * j;
      const float* skb = st;
      const float* svb = st + SB * D;
      float* sdb = const_cast<float*>(st) + SB * D * (comp ? 2 : 1);
      const int rb = k * SB, nbs = min(SB, nb - rb);
      if (SCORE && !dbulk && lane < nbs * r)  // r < 4: the Dbar rows by plain loads, 4 floats per row
        sdb[(lane / r) * 4 + lane % r] = __ldcg(a.dbar + (row0 + rb) * r + lane);
      if (!mbar_wait_bounded(bars + 2 * warp, usesK & 1u, a.status, s, h, 10)) {
        bad = true;
        break;
      }
      ++usesK;
      __syncwarp();
      // zbar partial dots of the stage's SB blocks and G heads
      float p[NV];
#pragma unroll
      for (int b = 0; b < SB; ++b) {
        float x[CPL];
        lds_vec<CPL>(skb + b * D + CPL * lane, x);
        if (b >= nbs) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) x[c] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float t = q[g][0] * x[0];
#pragma unroll
          for (int c = 1; c < CPL; ++c) t = fmaf(q[g][c], x[c], t);
          p[b * G + g] = t;
        }
      }
      butterfly<NV>(p, lane);
      const float zb = p[0];
      const bool ok = vb < nbs;
      const int gb = b0 + rb + vb;  // unit-local block of this lane's value
      const float cv = ok ? ln_count(gb == N - 1 ? L - kBlock * gb : kBlock) + zb : -INFINITY;
      float s2 = 0.f;
      if (SCORE) {
        if constexpr (RB) {
          // long Dbar rows (r = 32 RPL): lane holds Dbar and Qsq coordinates [RPL lane, RPL lane + RPL),
          // read as one RPL-float vector each (no bank conflicts)
          float ps[NV];
#pragma unroll
          for (int b = 0; b < SB; ++b) {
            float x[RPL];
            if (b < nbs) {  // (warp-uniform)
              lds_vec<RPL>(sdb + b * rs + RPL * lane, x);
            } else {
#pragma unroll
              for (int t = 0; t < RPL; ++t) x[t] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              float w[RPL];
              lds_vec<RPL>(sqw + g * rr + RPL * lane, w);
              float t = w[0] * x[0];
#pragma unroll
              for (int c = 1; c < RPL; ++c) t = fmaf(w[c], x[c], t);
              ps[b * G + g] = t;
            }
          }
          butterfly<NV>(ps, lane);
          s2 = ps[0] * (1.f / (float)D);
        } else {
          if (ok) {
            const float* drow = sdb + vb * rs;
            const float* qsr = sqw + vg * rr;
            float t = 0.f;
            if (r < 4) {
              // r = 1 or 2: the rows are padded to 4 floats and only the first r are written
              const float4 qv = *reinterpret_cast<const float4*>(qsr);
              const float4 dv = *reinterpret_cast<const float4*>(drow);
              t = r == 2 ? fmaf(qv.x, dv.x, qv.y * dv.y) : qv.x * dv.x;
            } else if (r <= 16) {
#pragma unroll
              for (int tt = 0; tt < 16; tt += 4) {
                if (tt < r) {
                  const float4 qv = *reinterpret_cast<const float4*>(qsr + tt);
                  const float4 dv = *reinterpret_cast<const float4*>(drow + tt);
                  t = fmaf(qv.x, dv.x, fmaf(qv.y, dv.y, fmaf(qv.z, dv.z, fmaf(qv.w, dv.w, t))));
                }
              }
            } else {
              for (int tt = 0; tt < r; tt += 4) {
                const float4 qv = *reinterpret_cast<const float4*>(qsr + tt);
                const float4 dv = *reinterpret_cast<const float4*>(drow + tt);
                t = fmaf(qv.x, dv.x, fmaf(qv.y, dv.y, fmaf(qv.z, dv.z, fmaf(qv.w, dv.w, t))));
              }
            }
            s2 = t * (1.f / (float)D);
          }
        }
      }
      if (primary && ok) {
        const int64_t o = (row0 + rb + vb) * Gp + vg;
        a.zs[o] = zb;
        if (SCORE) {
          a.ss[o] = s2;
          const float av = cv + ((a.variant & kVarFirstOrderMass) ? 0.f : 0.5f * s2);
          const float mn = fmaxf(lm, av);
          ll = (lm == -INFINITY ? 0.f : ll * __expf(lm - mn)) + __expf(av - mn);
          lm = mn;
        }
      }
      if (comp) {
        // the stage's maximum of ln|b| + zbar per head: lanes holding one head
        // differ in the bits outside [SH, SH + GB)
        float gm = cv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const bool head_bit = o >= (1 << SH) && o < (1 << (SH + GB));
          if (!head_bit) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
        }
        // every lane learns every head's stage maximum (from lane g << SH) and raises its references
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float m = __shfl_sync(0xffffffffu, gm, g << SH);
          if (m > ref[g]) {  // warp-uniform
            const float f = ref[g] == -INFINITY ? 0.f : __expf(ref[g] - m);
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[g][c] *= f;
            if (vg == g) wsl *= f;
            ref[g] = m;
          }
        }
        // the weight of this lane's value, then acc += w vbar over the stage's blocks
        float rg = ref[0];
#pragma unroll
        for (int g = 1; g < G; ++g)
          if (vg == g) rg = ref[g];
        const float w = ok ? __expf(cv - rg) : 0.f;
        if (primary) {
          swr[vb * G + vg] = w;
          wsl += w;
        }
      }
      __syncwarp();  // the kbar and Dbar rows are read (and the weights written): the next stage's may come
      if (lane == 0 && j + 1 < mine) issueK(k + kWarps);
      if (comp) {
        if (!mbar_wait_bounded(bars + 2 * warp + 1, usesV & 1u, a.status, s, h, 11)) {
          bad = true;
          break;
        }
        ++usesV;
        __syncwarp();
        for (int b = 0; b < nbs; ++b) {
          float x[CPL], wv[G];
          lds_vec<CPL>(svb + b * D + CPL * lane, x);
#pragma unroll
          for (int g = 0; g < G; ++g) wv[g] = swr[b * G + g];
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[g][c] = fmaf(wv[g], x[c], acc[g][c]);
        }
        __syncwarp();  // the vbar rows and the weights are read
        if (lane == 0 && j + 1 < mine) issueV(k + kWarps);
      }
    }
    if (bad) {
      mbar_drain_bounded(bars + 2 * warp);
      mbar_drain_bounded(bars + 2 * warp + 1);
      if (lane == 0) *sbad = 1;
    }
    __syncthreads();  // every stage of the segment is consumed: the slots are free
    if (TRACE && !nseg_done) t_first = global_ns();
    ++nseg_done;
    if (*sbad) break;  // a copy never arrived: this CTA stops (the status word holds the timeout)

    // ---- the segment's record: the warps' parts per head combined through the slots
    // (this runs once per segment: short dependency chains, all heads at once)
    float* xr = slots;                   // [kWarps][G][4]
    float* xa = slots + kWarps * G * 4;  // [kWarps][G][D]
    {
      // lanes holding one head differ in the lane bits outside [SH, SH + GB): reduce over those
      float m = primary ? lm : -INFINITY, l = primary ? ll : 0.f, w = primary ? wsl : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        if (o >= (1 << SH) && o < (1 << (SH + GB))) continue;
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
        lse_merge(m, l, m2, l2);
        w += __shfl_xor_sync(0xffffffffu, w, o);
      }
      if ((lane & ~(((1 << GB) - 1) << SH)) == 0) {  // lane vg << SH holds head vg
        float rg = ref[0];
#pragma unroll
        for (int gg = 1; gg < G; ++gg)
          if (vg == gg) rg = ref[gg];
        *reinterpret_cast<float4*>(xr + (warp * G + vg) * 4) = make_float4(m, l, rg, w);
      }
    }
    if (comp)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < CPL; ++c) xa[(warp * G + g) * D + CPL * lane + c] = acc[g][c];
    if (TRACE && nseg_done == 1) t_r1 = global_ns();
    __syncthreads();
    if (TRACE && nseg_done == 1) t_r2 = global_ns();
    if (warp < G) {
      const int g = warp;
      // lane w < kWarps takes warp w's part; three xor steps combine them
      float4 e = lane < kWarps ? *reinterpret_cast<const float4*>(xr + (lane * G + g) * 4)
                               : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      float M = e.x, Ls = e.y, R = e.z;
#pragma unroll
      for (int o = 1; o < kWarps; o <<= 1) {
        const float M2 = __shfl_xor_sync(0xffffffffu, M, o), L2 = __shfl_xor_sync(0xffffffffu, Ls, o);
        lse_merge(M, Ls, M2, L2);
        R = fmaxf(R, __shfl_xor_sync(0xffffffffu, R, o));
      }
      float fw = (lane < kWarps && e.z != -INFINITY) ? __expf(e.z - R) : 0.f;
      float Ws = lane < kWarps ? e.w * fw : 0.f;
#pragma unroll
      for (int o = 1; o < kWarps; o <<= 1) Ws += __shfl_xor_sync(0xffffffffu, Ws, o);
      float o[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) o[c] = 0.f;
      if (comp)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = __shfl_sync(0xffffffffu, fw, w);
#pragma unroll
          for (int c = 0; c < CPL; ++c) o[c] = fmaf(xa[(w * G + g) * D + CPL * lane + c], f, o[c]);
        }
      if (lane == 0) a.rec[(int64_t)si * G + g] = make_float4(M, Ls, comp ? R : -INFINITY, comp ? Ws : 0.f);
      if (comp) {
        float* dst = a.comp + ((int64_t)si * G + g) * D + CPL * lane;
        if constexpr (CPL == 4)
          *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        else
          *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
      }
    }
    if (TRACE && nseg_done == 1) t_r3 = global_ns();
    __syncthreads();  // the slots are free for the next segment
  }
  if (TRACE && threadIdx.x == 0 && (int)blockIdx.x < a.trace_cap) {
    unsigned long long* rr = a.trace + 1 + 8 * (int64_t)blockIdx.x;
    rr[0] = ((unsigned long long)blockIdx.x << 32) | (unsigned)nseg_done;
    rr[1] = 0ull;
    rr[2] = t_start;
    rr[3] = t_plan;
    rr[4] = t_first;
    rr[5] = global_ns();
    rr[6] = t_r1 - t_first;
    rr[7] = ((t_r2 - t_r1) << 32) | (t_r3 - t_r2);
  }
}

template <int D, int G, int MODE, bool TRACE>
static const void* stream_fn_t(int r) {
  if constexpr (D >= 128)
    if (r >= 128) return reinterpret_cast<const void*>(&k_stream<D, G, MODE, 4, 4, TRACE>);
  if (long_dbar(r)) return reinterpret_cast<const void*>(&k_stream<D, G, MODE, 4, 2, TRACE>);
  return reinterpret_cast<const void*>(&k_stream<D, G, MODE, (G >= 8 ? 4 : 8), 0, TRACE>);
}
template <int D, int G, int MODE>
static const void* stream_fn(int r, bool trace = false) {
  return trace ? stream_fn_t<D, G, MODE, true>(r) : stream_fn_t<D, G, MODE, false>(r);
}

template <int D, int G, int MODE>
static cudaError_t launch_stream_mode(const LayerArgs& a, cudaStream_t st, bool pdl) {
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  const void* fn = stream_fn<D, G, MODE>(a.r, a.trace != nullptr);
  const size_t smem = (size_t)stream_smem_bytes(D, a.r, G, SCORE, COMP);  // (limit raised by prepare_stream)
  LayerArgs args = a;
  chain_split(args, MODE);
  void* argv[] = {&args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(args.Q + args.P));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, argv);
}

template <int D, int G>
static int ctas_per_sm_dg(int r) {
  const void* fn = stream_fn<D, G, kFusedDecode>(r);
  const int smem = stream_smem_bytes(D, r, G, true, true);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, (size_t)smem) != cudaSuccess) return 1;
  return n;
}

int stream_ctas_per_sm(int D, int r, int G) {
  if (D == 128) {
    switch (G) {
      case 1: return ctas_per_sm_dg<128, 1>(r);
      case 2: return ctas_per_sm_dg<128, 2>(r);
      case 4: return ctas_per_sm_dg<128, 4>(r);
      default: return ctas_per_sm_dg<128, 8>(r);
    }
  }
  switch (G) {
    case 1: return ctas_per_sm_dg<64, 1>(r);
    case 2: return ctas_per_sm_dg<64, 2>(r);
    case 4: return ctas_per_sm_dg<64, 4>(r);
    default: return ctas_per_sm_dg<64, 8>(r);
  }
}

template <int D, int G>
static cudaError_t launch_stream_dg(const LayerArgs& a, int mode, cudaStream_t st, bool pdl) {
  switch (mode) {
    case kFusedDecode: return launch_stream_mode<D, G, kFusedDecode>(a, st, pdl);
    case kFusedScoreSelect: return launch_stream_mode<D, G, kFusedScoreSelect>(a, st, pdl);
    case kFusedAttend: return launch_stream_mode<D, G, kFusedAttend>(a, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_stream(const LayerArgs& a, int mode, cudaStream_t st, bool pdl) {
#define COMPKV_G(DD)                                          \
  switch (a.G) {                                              \
    case 1: return launch_stream_dg<DD, 1>(a, mode, st, pdl); \
    case 2: return launch_stream_dg<DD, 2>(a, mode, st, pdl); \
    case 4: return launch_stream_dg<DD, 4>(a, mode, st, pdl); \
    case 8: return launch_stream_dg<DD, 8>(a, mode, st, pdl); \
    default: return cudaErrorInvalidValue;                    \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

size_t stream_smem(int D, int r, int G) { return (size_t)stream_smem_bytes(D, r, G, true, true); }

template <int D, int G, int MODE>
static cudaError_t prepare_stream_mode(int r) {
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  const int smem = stream_smem_bytes(D, r, G, SCORE, COMP);
  cudaError_t e = raise_smem_limit(stream_fn<D, G, MODE>(r, false), smem);
  if (e == cudaSuccess) e = raise_smem_limit(stream_fn<D, G, MODE>(r, true), smem);
  return e;
}

template <int D, int G>
static cudaError_t prepare_stream_dg(int r) {
  cudaError_t e = prepare_stream_mode<D, G, kFusedDecode>(r);
  if (e == cudaSuccess) e = prepare_stream_mode<D, G, kFusedScoreSelect>(r);
  if (e == cudaSuccess) e = prepare_stream_mode<D, G, kFusedAttend>(r);
  return e;
}

cudaError_t prepare_stream(int D, int r, int G) {
#define COMPKV_G(DD)                             \
  switch (G) {                                   \
    case 1: return prepare_stream_dg<DD, 1>(r);  \
    case 2: return prepare_stream_dg<DD, 2>(r);  \
    case 4: return prepare_stream_dg<DD, 4>(r);  \
    case 8: return prepare_stream_dg<DD, 8>(r);  \
    default: return cudaErrorInvalidValue;       \
  }
  if (D == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

}  // namespace compkv
