// Selection, exact attention and Mean compensation of the CompKV decode step
// (onedev.kr/papers/157), after the summary stream (stream_kernel.cu).
//
// One thread-block cluster of C CTAs per (sequence, KV head) unit.  CTA rank p
// owns the unit's blocks [p bpc, (p + 1) bpc) (bpc = ceil(N / C) rounded up
// to 4) and, of the stream's segment records, those with index = p (mod C).
//   a. After the stream: warp 0 merges the unit's segment records and the
//      open block's a_g (which the stream kernel recomputed) into LSE_g, and
//      warp 1 copies the CTA's zbar and sigma2 rows.
//   b. S_b = sum_g phat_{g,b} sigma2_{g,b} ("무엇과 다른가") of the CTA's blocks
//      as order-preserving keys and a 12-bit histogram of the candidates
//      1..N-3.  After a cluster barrier, warp 0 of every CTA reads the peers'
//      counts in three levels of 16 bins and finds the threshold bin T where
//      the count of larger keys reaches K - 3 (the forced sink block and the
//      two most recent blocks take the other three places of the budget).
//   c. Blocks above T, and the forced ones, are selected for sure: each CTA
//      lists its own in ascending order, and the keys of its blocks in T,
//      for the peers to read after a second cluster barrier.  Its warps start
//      on the top eight of its own list before that barrier completes.
//   d. After the barrier every CTA reads the peers' counts and tie lists,
//      ranks the keys in T (ties to the lower block index) and spreads the
//      rest of the work -- own lists longer than eight and the tie winners --
//      over the warps left idle, in one order that every CTA derives alike.
//   e. A warp attends exactly to one block's bf16 K/V at a time with
//      tensor-core products (q and the probabilities split into bf16 high and
//      low parts, fp32 accumulation) and removes the block's own
//      Mean-compensation term, which the stream added for every block
//      ("어떻게 동작하나": unselected blocks contribute |b| e^{zbar} vbar and
//      |b| e^{zbar}); the partials and the CTA's share of the compensation
//      sums merge across the cluster into out = acc / l.
// By Jensen, sum_{j in b} e^{z_j} >= |b| e^{zbar_b}, so removing a selected
// block's mean term never makes a block's net weight negative.  If every
// block is selected there is no compensation (the step is dense attention).
#include "compkv_launch.h"
#include "decode_common.cuh"

namespace compkv {

constexpr int kPW = 8;                // warps of a post CTA
constexpr int kPT = 32 * kPW;
constexpr int kTieCap = 64;           // tie entries one CTA may push
constexpr int kRankMax = 256;         // tie entries ranked directly
constexpr int kDigitShift = 19;       // level-0 digit: key bits 30..19 (exponent + 4 mantissa bits)
constexpr int kFine = 4096;

template <int D>
struct InvSqrtP;
template <>
struct InvSqrtP<64> {
  static constexpr float v = 0.125f;
};
template <>
struct InvSqrtP<128> {
  static constexpr float v = 0.08838834764831845f;
};

// Attention staging of one warp, 1024-byte aligned: the block's 16 K rows, then
// its 16 V rows, each as D / 64 boxes of 16 rows x 128 bytes written by the
// tensor copy with the 128-byte swizzle (16-byte chunk c of row t lies at
// chunk c ^ (t % 8), so the eight rows one ldmatrix reads fall in eight
// different bank quads), then vbar of the block (fp32 [D]).
__host__ __device__ constexpr int stg_kv(int D) { return kBlock * 2 * D; }  // bytes of the K (or V) boxes
__host__ __device__ constexpr int stg_bytes(int D) { return (2 * stg_kv(D) + 4 * D + 1023) & ~1023; }

// Shared memory of the post kernel, in 4-byte words.
struct PostLayout {
  int zsl, ssl, stg, red, keys, own, csh, qf, plan, anm, lsep, hf, tie, dense, xexp, xfine, xref, lh, xm, win, misc,
      bars, total;
};
__host__ __device__ inline int post_items(int D, int G) { return G * D / 4; }
__host__ __device__ inline int post_ipr(int D, int G, int C) { return (post_items(D, G) + C - 1) / C; }
__host__ __device__ inline PostLayout post_layout(int D, int G, int C, int bpc_max, int K) {
  PostLayout l;
  const int Gp = pad_g(G);
  int o = 0;
  // union: zbar and sigma2 of the CTA's blocks (keys) | attention staging | the warps' partials
  l.zsl = o;
  l.ssl = o + bpc_max * Gp;
  l.stg = o;
  l.red = o;
  const int zw = 2 * bpc_max * Gp;
  const int sw = kPW * stg_bytes(D) / 4 + 256;  // (+ 1 KB to align the staging to 1024 bytes)
  const int rw = kPW * D * 8 + 2 * kPW * 8;  // [kPW][D][8] partial numerators, [kPW][8] maxima and sums
  int uw = zw > sw ? zw : sw;
  uw = uw > rw ? uw : rw;
  o += (uw + 3) & ~3;
  l.keys = o; o += (bpc_max + 3) & ~3;
  l.own = o; o += ((bpc_max < K ? bpc_max : K) + 3) & ~3;
  l.csh = o; o += G * D;               // this CTA's share of the compensation numerator [G][D]
  l.qf = o; o += (D / 16) * 32 * 4;    // q fragments of every lane, per k-step (uint4)
  l.plan = o; o += 3 * kMaxBatch + 4;  // tokens, streamed blocks and first segment of every sequence
  l.anm = o; o += kMaxG;               // a_g of the open block
  l.lsep = o; o += 2 * kMaxG;          // (max, sum) of the records' logsumexp per head
  // selection: the local fine histogram [4096] (read by the peers until barrier 2); after
  // barrier 2, the dense copy of the cluster's tie lists (or, on the rare path, the selection bitmap)
  l.hf = o;
  l.tie = o;
  l.dense = o + 2 * kMaxC * kTieCap;
  o += kFine;
  l.xexp = o; o += 256;                            // this CTA's counts per 8-bit key prefix (the exponent)
  l.xfine = o; o += 16 + 2 * kTieCap;              // counts per 4-bit prefix [16]; this CTA's tie list [kTieCap]
  l.xref = o; o += 3 * 256;                        // refinement histograms (rank 0)
  l.lh = o; o += 256;                              // refinement local histogram
  l.xm = o; o += post_ipr(D, G, C) * C * 8;        // merge staging: [items per rank][C][acc4, m, l, -, -]
  l.win = o; o += kRankMax + 4;                    // tie winners in rank order (before: local tie indices)
  l.misc = o; o += 192;
  l.bars = o; o += 2 * (kPW + 2);
  l.total = o;
  return l;
}

// misc slots (ints unless noted)
enum : int {
  kMT = 0, kMAbove, kMCntT, kMNtie, kMOwn, kMBad, kMTot,
  kMWT = 8,          // [8] warp totals of the own-list scan
  kMCR = 24,         // float [8]: compensation reference of this CTA's share
  kMCW = 32,         // float [8]: compensation weight sum of the share
  kMCnt = 40,        // int2 [16]: per CTA (own selected count, tie count), pushed by the peers
  kMCntR = 72,       // int [16]: refinement counts, pushed by the peers
  kMScan = 88,       // int [8]: scan scratch
  kMPlan = 96,       // blocks per segment
  kMFits = 100,      // [2] bit s: sequence s had room for its token
  kMCntA = 104,      // int [16]: rare path, every CTA's final own count
  kMR0 = 120,        // int [8]: rare path, the block each warp attended before the exchange
  kMTpre = 128,      // int [16]: exclusive prefix of the CTAs' tie counts
  kMMine = 160,      // int [2]: this CTA's own-list count and tie count (read by the peers)
  kMTcnt = 168,      // int [16]: the CTAs' tie counts
};

// ---------------------------------------------------------------- tensor-core pieces
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// d += A (16 x 16, row) * B (16 x 8, col), bf16 inputs, fp32 accumulation
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// (x, y) as bf16x2 high parts and the bf16x2 of what they leave (x first, in the low half)
__device__ __forceinline__ void split_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(hv);
  const __nv_bfloat162 lv = __floats2bfloat162_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&hv);
  lo = *reinterpret_cast<const uint32_t*>(&lv);
}

// One block of exact attention for the warp's running state.  Lane (r, c) =
// (lane / 4, lane % 4).  Scores S^T = q K^T as a 16 x 16 product (rows: the
// query heads, zero beyond G; columns: the 16 tokens), so lane (r, c) holds
// head r at tokens 2c, 2c+1, 8+2c, 9+2c -- which is also its fragment of the
// probabilities as the B operand of O^T += V^T P (rows: coordinates, columns:
// heads).  m, l: head r (every lane of the quad alike).  acc[mt]: O^T at
// coordinates 16 mt + r (+ 8) for heads 2c, 2c + 1.  With `cb`, the block's
// compensation term |b| e^{zbar} (zb: zbar of head r) and its vbar (staged
// after the V rows) come off, in the same rescale.
template <int D, int G>
__device__ __forceinline__ void blk_attend(float& m, float& l, float (&acc)[D / 16][4], const uint4* qf,
                                           const char* stg, int n, bool cb, float zb, int lane) {
  constexpr int KS = D / 16;
  const int r = lane >> 2, c = lane & 3;
  // ldmatrix rows: matrix lane / 8 = (tokens 0-7 | 8-15) x (coordinates +0 | +8); the row's
  // 16-byte chunk 2 ks + hb of k-step ks lies in box ks / 4 at swizzled chunk ((2 ks + hb) % 8) ^ (t % 8)
  const int t = (lane >> 4) * 8 + (lane & 7), hb = (lane >> 3) & 1, swz = t & 7;
  const uint32_t kaddr = smem_u32(stg) + (uint32_t)t * 128u;
  const uint32_t vaddr = kaddr + (uint32_t)stg_kv(D);
  auto chunk = [&](int ks) -> uint32_t {
    return (uint32_t)((ks >> 2) * (kBlock * 128) + ((((2 * ks) & 7) + hb) ^ swz) * 16);
  };
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4(kaddr + chunk(ks), b0, b1, b2, b3);
    const uint4 qv = qf[ks * 32 + lane];  // high parts (k 2c.., k 8+2c..), low parts
    mma_bf16(s0, qv.x, 0u, qv.y, 0u, b0, b1);
    mma_bf16(s1, qv.x, 0u, qv.y, 0u, b2, b3);
    mma_bf16(s0, qv.z, 0u, qv.w, 0u, b0, b1);
    mma_bf16(s1, qv.z, 0u, qv.w, 0u, b2, b3);
  }
  const float x0 = 2 * c < n ? s0[0] : -INFINITY, x1 = 2 * c + 1 < n ? s0[1] : -INFINITY;
  const float x2 = 8 + 2 * c < n ? s1[0] : -INFINITY, x3 = 9 + 2 * c < n ? s1[1] : -INFINITY;
  float bm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
  bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
  const bool live = r < G;
  const float e = (cb && live) ? ln_count(n) + zb : -INFINITY;
  const float mn = fmaxf(m, fmaxf(bm, e));
  const float fo = m == -INFINITY ? 0.f : __expf(m - mn);
  const float fn = (cb && live) ? __expf(e - mn) : 0.f;
  const float p0 = live ? __expf(x0 - mn) : 0.f, p1 = live ? __expf(x1 - mn) : 0.f;
  const float p2 = live ? __expf(x2 - mn) : 0.f, p3 = live ? __expf(x3 - mn) : 0.f;
  float ps = (p0 + p1) + (p2 + p3);
  ps += __shfl_xor_sync(0xffffffffu, ps, 1);
  ps += __shfl_xor_sync(0xffffffffu, ps, 2);
  l = l * fo + ps - fn;
  m = mn;
  // the factors of this lane's accumulator columns (heads 2c, 2c+1 live in quads 2c, 2c+1)
  const float foA = __shfl_sync(0xffffffffu, fo, 8 * c), foB = __shfl_sync(0xffffffffu, fo, 8 * c + 4);
  const float fnA = __shfl_sync(0xffffffffu, fn, 8 * c), fnB = __shfl_sync(0xffffffffu, fn, 8 * c + 4);
  uint32_t ph0, pl0, ph1, pl1;
  split_bf16(p0, p1, ph0, pl0);
  split_bf16(p2, p3, ph1, pl1);
  const float* vb = reinterpret_cast<const float*>(stg + 2 * stg_kv(D));
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const float v0 = cb ? vb[16 * mt + r] : 0.f, v1 = cb ? vb[16 * mt + 8 + r] : 0.f;
    acc[mt][0] = fmaf(acc[mt][0], foA, -fnA * v0);
    acc[mt][1] = fmaf(acc[mt][1], foB, -fnB * v0);
    acc[mt][2] = fmaf(acc[mt][2], foA, -fnA * v1);
    acc[mt][3] = fmaf(acc[mt][3], foB, -fnB * v1);
    uint32_t a0, a1, a2, a3;
    ldsm_x4_t(vaddr + chunk(mt), a0, a1, a2, a3);
    mma_bf16(acc[mt], a0, a1, a2, a3, ph0, ph1);
    mma_bf16(acc[mt], a0, a1, a2, a3, pl0, pl1);
  }
}

// ---------------------------------------------------------------- the phases
// The code of this kernel runs once per call on every multiprocessor it
// occupies, so its instruction footprint is on the critical path: loops over
// runtime counts stay rolled, and every piece of work has one call site.

// LSE_g = logsumexp of a_g over the unit's blocks, from its nseg segment records (and the open
// block's a_g), by one warp: lane j merges records of head j % G; lanes of one head then merge
// across the warp; lane g < G writes LSE_g.
template <int G>
__device__ __forceinline__ void record_lse(const LayerArgs& a, int i0, int nseg, float an, bool app, float* lsep,
                                           int lane) {
  float M = -INFINITY, S = 0.f;
  const int tot = nseg * G;
  const float4* base = a.rec + (int64_t)i0 * G;
#pragma unroll 1
  for (int k0 = 0; k0 < tot; k0 += 256) {  // eight records per lane in flight at once
    float4 e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = k0 + lane + 32 * j;
      e[j] = idx < tot ? __ldcg(base + idx) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    }
    // the eight parts at their common maximum: independent exponentials instead of a chain of merges
    float mc = e[0].x;
#pragma unroll
    for (int j = 1; j < 8; ++j) mc = fmaxf(mc, e[j].x);
    float sc = 0.f;
    if (mc != -INFINITY) {
#pragma unroll
      for (int j = 0; j < 8; ++j) sc += e[j].x == -INFINITY ? 0.f : e[j].y * __expf(e[j].x - mc);
    }
    lse_merge(M, S, mc, sc);
  }
  // across the lanes of a head: the maximum, then the sums rescaled to it
  float Mw = M;
#pragma unroll
  for (int o = G; o < 32; o <<= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, o));
  float Sw = M == -INFINITY ? 0.f : S * __expf(M - Mw);
#pragma unroll
  for (int o = G; o < 32; o <<= 1) Sw += __shfl_xor_sync(0xffffffffu, Sw, o);
  if (lane < G) {  // LSE_g, with the open block's a_g (`an`, lane g) when this call appended
    if (app) lse_merge(Mw, Sw, an, 1.f);
    lsep[lane] = Mw + __logf(Sw);
  }
}

// This CTA's share of the compensation sums: segment records p, p + C, ...
// rescaled to their common maximum; thread items (head, column quad), every
// load of an item issued before any is used.
template <int D, int G>
__device__ __forceinline__ void comp_share(const LayerArgs& a, int i0, int nseg, int p, int C, float* csh, float* cR,
                                           float* cW, int t, int nt) {
  const int nk = p < nseg ? (nseg - 1 - p) / C + 1 : 0;
#pragma unroll 1
  for (int i4 = t; i4 < G * D / 4; i4 += nt) {
    const int g = i4 / (D / 4), col = 4 * (i4 % (D / 4));
    float R = -INFINITY, Wsum = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int k0 = 0; k0 < nk; k0 += 4) {
      float4 e[4], v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rec = i0 + p + C * (k0 + j);
        const bool ok = k0 + j < nk;
        e[j] = ok ? __ldcg(a.rec + (int64_t)rec * G + g) : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        v[j] = ok ? __ldcg(reinterpret_cast<const float4*>(a.comp + ((int64_t)rec * G + g) * D + col))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (e[j].z == -INFINITY) continue;
        const float mn = fmaxf(R, e[j].z);
        const float fo = R == -INFINITY ? 0.f : __expf(R - mn);
        const float fn = __expf(e[j].z - mn);
        A.x = A.x * fo + v[j].x * fn;
        A.y = A.y * fo + v[j].y * fn;
        A.z = A.z * fo + v[j].z * fn;
        A.w = A.w * fo + v[j].w * fn;
        Wsum = Wsum * fo + e[j].w * fn;
        R = mn;
      }
    }
    *reinterpret_cast<float4*>(csh + g * D + col) = A;
    if (col == 0) {
      cR[g] = R;
      cW[g] = Wsum;
    }
  }
}

// Exclusive prefix of `v` over the CTA's kPT threads; `total` receives the
// sum.  Two CTA barriers.
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
#pragma unroll 1
  for (int w = 0; w < kPW; ++w) {
    const int t = scratch[w];
    base += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// Warp 0: the ascending list of the set bits of words[0..nw) (bit i = block
// lo + i) into list[0..cap), returns the count (in warp 0).
__device__ __noinline__ int bitmap_list(const unsigned* words, int nw, int lo, int* list, int cap, int lane) {
  const int per = (nw + 31) / 32;
  int loc = 0;
#pragma unroll 1
  for (int k = 0; k < per; ++k) {
    const int w = per * lane + k;
    if (w < nw) loc += __popc(words[w]);
  }
  int incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - loc;
#pragma unroll 1
  for (int k = 0; k < per; ++k) {
    const int w = per * lane + k;
    if (w < nw) {
      unsigned word = words[w];
      while (word) {
        const int bit = __ffs(word) - 1;
        if (run < cap) list[run] = lo + 32 * w + bit;
        ++run;
        word &= word - 1u;
      }
    }
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// One level of the cluster-wide threshold search, by one warp.  The 16 counts at
// `cnt` (the same shared-memory offset in every CTA of the cluster) are summed
// over the C CTAs -- lane q < C reads CTA q's, a halving butterfly leaves the
// total of bin l >> 1 in lane l -- and the bin where the count of larger keys,
// added to `run`, reaches `need` is returned as x, with the count above that
// bin (including `run`) as y and its own count as z.
__device__ __noinline__ int3 cluster_level(const uint32_t* cnt, int C, int lane, int need, int run) {
  uint32_t v[16];
  if (lane < C) {
    const uint32_t src = peer_smem(cnt, (uint32_t)lane);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 x = ld_peer_u4(src + 16u * k);
      v[4 * k] = x.x;
      v[4 * k + 1] = x.y;
      v[4 * k + 2] = x.z;
      v[4 * k + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = 0u;
  }
#pragma unroll
  for (int o = 16, nv = 16; o >= 2; o >>= 1, nv >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < nv / 2) {
        const uint32_t send = up ? v[i] : v[i + nv / 2];
        const uint32_t keep = up ? v[i + nv / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  const uint32_t tot = v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);  // bin lane >> 1
  // count of the bins at and above lane >> 1 (even lanes carry their bin once)
  uint32_t sfx = (lane & 1) ? 0u : tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, sfx, o);
    if (lane + o < 32) sfx += y;
  }
  const int above = run + (int)(sfx - tot);
  const bool hit = !(lane & 1) && above < need && need <= above + (int)tot;
  const int src = __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
  return make_int3(src >> 1, __shfl_sync(0xffffffffu, above, src), (int)__shfl_sync(0xffffffffu, tot, src));
}

// Rare path of the selection: more keys share the threshold bin T than the
// tie lists hold.  The keys in play (candidates in bin T) are resolved by
// three more radix digits (bits 18..11, 10..3, 2..0), each a histogram summed
// at rank 0 with one cluster barrier, and keys equal in every bit go to the
// lowest block indices (counts exchanged, one more barrier).  Sets the bits of
// the selected in-play blocks in `bits` (which holds the sure blocks on
// entry).  Called by every thread of every CTA of the cluster.
__device__ __noinline__ void refine_select(const uint32_t* keys, unsigned* bits, int nown, int b_lo, int N, uint32_t T,
                                           int need, uint32_t* xref, uint32_t* lh, int* misc, int C, int p) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t pfx = T << kDigitShift, pm = 0xFFFFFFFFu << kDigitShift;
  bool done = false;
#pragma unroll 1
  for (int level = 1; level <= 3 && !done; ++level) {
    const int shift = level == 1 ? 11 : (level == 2 ? 3 : 0);
    const int nb = level == 3 ? 8 : 256;
    const uint32_t dm = (uint32_t)nb - 1u;
#pragma unroll 1
    for (int i = tid; i < 256; i += kPT) lh[i] = 0u;
    __syncthreads();
#pragma unroll 1
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      if (b < 1 || b > N - 3) continue;
      const uint32_t key = keys[i];
      if ((key & pm) == pfx && !((bits[i >> 5] >> (i & 31)) & 1u)) atomicAdd(&lh[(key >> shift) & dm], 1u);
    }
    __syncthreads();
    uint32_t* xr = xref + (level - 1) * 256;
#pragma unroll 1
    for (int i = tid; i < nb; i += kPT)
      if (lh[i]) red_peer_add(peer_smem(xr + i, 0), lh[i]);
    cluster_sync_all();
    // the digit where the count of larger in-play keys reaches `need` (thread t: digit nb - 1 - t)
    int c = 0;
    if (tid < nb) c = (int)ld_peer_u32(peer_smem(xr + (nb - 1 - tid), 0));
    int tot;
    const int before = cta_exclusive_scan(c, misc + kMScan, &tot, lane, warp);
    if (tid < nb && before < need && need <= before + c) {
      misc[kMT] = nb - 1 - tid;
      misc[kMAbove] = before;
      misc[kMCntT] = c;
    }
    __syncthreads();
    const uint32_t Dg = (uint32_t)misc[kMT];
    const int above = misc[kMAbove], cnt = misc[kMCntT];
    const bool all = cnt == need - above;
#pragma unroll 1
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      if (b < 1 || b > N - 3) continue;
      const uint32_t key = keys[i];
      if ((key & pm) != pfx || ((bits[i >> 5] >> (i & 31)) & 1u)) continue;
      const uint32_t dg = (key >> shift) & dm;
      if (dg > Dg || (all && dg == Dg)) atomicOr(&bits[i >> 5], 1u << (i & 31));
    }
    need -= above;
    pfx |= Dg << shift;
    pm |= dm << shift;
    done = all;
    __syncthreads();
  }
  if (!done) {
    // keys equal in every bit: the `need` lowest block indices of the cluster
    int c = 0;
#pragma unroll 1
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      if (b < 1 || b > N - 3) continue;
      if ((keys[i] & pm) == pfx && !((bits[i >> 5] >> (i & 31)) & 1u)) ++c;
    }
    int tot;
    cta_exclusive_scan(c, misc + kMScan, &tot, lane, warp);
    if (tid < C) st_peer_u32(peer_smem(misc + kMCntR + p, (uint32_t)tid), (uint32_t)tot);
    cluster_sync_all();
    int before = 0;
#pragma unroll 1
    for (int q = 0; q < p; ++q) before += misc[kMCntR + q];
    int take = need - before;
    take = take < 0 ? 0 : (take > tot ? tot : take);
    if (tid == 0 && take > 0) {
      // the first `take` in-play blocks in index order: one thread scans
      int got = 0;
#pragma unroll 1
      for (int i = 0; i < nown && got < take; ++i) {
        const int b = b_lo + i;
        if (b < 1 || b > N - 3) continue;
        if ((keys[i] & pm) == pfx && !((bits[i >> 5] >> (i & 31)) & 1u)) {
          bits[i >> 5] |= 1u << (i & 31);
          ++got;
        }
      }
    }
    __syncthreads();
  }
}

// A block's K and V rows by 16-byte asynchronous copies of every lane into their swizzled places
// (K and V in host memory, or no tensor maps), out of line: the tensor copies are the common case.
template <int D>
__device__ __noinline__ void plain_copy(char* stg, const char* kg, const char* vg, int n, int lane) {
#pragma unroll 1
  for (int x = lane; x < n * (D / 8); x += 32) {
    const int t = x / (D / 8), j = x % (D / 8);
    const int so = (j >> 3) * kBlock * 128 + t * 128 + (((j & 7) ^ (t & 7)) << 4);
    cp_async16(stg + so, kg + x * 16);
    cp_async16(stg + stg_kv(D) + so, vg + x * 16);
  }
  cp_async_commit();
}

// The rare path as a whole (more candidates share bin T than the tie lists hold), by every
// thread of every CTA of the cluster, out of line so that its code stays out of the common
// path's: the own list with the sure blocks, refined by more radix digits (refine_select)
// and listed again; the CTAs' counts exchanged.  Returns (own count, this CTA's offset in the
// ascending selection, the selection's size).
__device__ __noinline__ int3 rare_select(const uint32_t* keys, unsigned* bits, int* own, int n_own, int nown, int b_lo,
                                         int N, int K, uint32_t T, int need, uint32_t* xref, uint32_t* lh, int* misc,
                                         int C, int p) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwo = (nown + 31) / 32;
#pragma unroll 1
  for (int w = tid; w < nwo; w += kPT) bits[w] = 0u;
  __syncthreads();
#pragma unroll 1
  for (int e = tid; e < n_own; e += kPT) atomicOr(&bits[(own[e] - b_lo) >> 5], 1u << ((own[e] - b_lo) & 31));
  __syncthreads();
  refine_select(keys, bits, nown, b_lo, N, T, need, xref, lh, misc, C, p);
  if (warp == 0) {
    const int nl = bitmap_list(bits, nwo, b_lo, own, nown < K ? nown : K, lane);
    if (lane == 0) misc[kMOwn] = nl;
  }
  __syncthreads();
  n_own = min(misc[kMOwn], nown < K ? nown : K);
  if (tid < C) st_peer_u32(peer_smem(misc + kMCntA + p, (uint32_t)tid), (uint32_t)n_own);
  cluster_sync_all();
  int before = 0, all = 0;
#pragma unroll 1
  for (int q = 0; q < C; ++q) {
    before += q < p ? misc[kMCntA + q] : 0;
    all += misc[kMCntA + q];
  }
  return make_int3(n_own, before, all);
}

// TRACE: the work-item trace is recorded (a.trace is set); the instance without it carries no
// trace code, which matters here because this kernel's code runs once per call.
template <int D, int G, int MODE, bool TRACE>
__global__ void __launch_bounds__(kPT, 2) k_post(const __grid_constant__ LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool ATT = (MODE & kFAttend) != 0;
  constexpr int KS = D / 16;
  extern __shared__ __align__(16) float psm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = a.C;
  const int u = blockIdx.x / C;
  const int p = (int)cluster_rank();
  const int s = u / a.Hkv, h = u % a.Hkv;
  const int K = a.K;
  const int Gp = pad_g(G);
  const PostLayout lay = post_layout(D, G, C, a.bpc_max, K);
  float* zsl = psm + lay.zsl;
  float* ssl = psm + lay.ssl;
  uint32_t* keys = reinterpret_cast<uint32_t*>(psm + lay.keys);
  int* own = reinterpret_cast<int*>(psm + lay.own);
  uint32_t* hf = reinterpret_cast<uint32_t*>(psm + lay.hf);
  uint2* dense = reinterpret_cast<uint2*>(psm + lay.dense);
  uint32_t* xexp = reinterpret_cast<uint32_t*>(psm + lay.xexp);
  uint32_t* xfine = reinterpret_cast<uint32_t*>(psm + lay.xfine);
  uint32_t* xref = reinterpret_cast<uint32_t*>(psm + lay.xref);
  uint32_t* lh = reinterpret_cast<uint32_t*>(psm + lay.lh);
  float* xm = psm + lay.xm;
  int* win = reinterpret_cast<int*>(psm + lay.win);
  int* misc = reinterpret_cast<int*>(psm + lay.misc);
  float* cR = reinterpret_cast<float*>(misc + kMCR);
  float* cW = reinterpret_cast<float*>(misc + kMCW);
  float* lsep = psm + lay.lsep;
  float* csh = psm + lay.csh;
  uint64_t* bars = reinterpret_cast<uint64_t*>(psm + lay.bars);  // [kPW] attention, [1] zbar/sigma2 copy
  const unsigned long long t_start = TRACE ? global_ns() : 0ull;
  unsigned long long t_wait = 0ull;

  // phase marks of the work-item trace: mark k goes to record 1 + k / 7, slot 1 + k % 7
  // (kept in shared memory until the end, so that no global store waits in a fence)
  __shared__ unsigned long long tmk[35];
  if (TRACE && tid < 35) tmk[tid] = 0ull;
  auto markt = [&](int k, int t) {
    if (TRACE && tid == t) tmk[k] = global_ns();
  };
  auto mark = [&](int k) { markt(k, 0); };

  // ---- set-up before the stream's results are visible; its global loads are issued together here
  const int Lold_s = __ldcg(a.seq_len + s);
  int sl0 = 0, sl1 = 0;
  if (warp == 0) {
    if (lane < a.B) sl0 = __ldcg(a.seq_len + lane);
    if (lane + 32 < a.B) sl1 = __ldcg(a.seq_len + lane + 32);
  }
  const float* qunit = a.q + ((int64_t)s * a.Hkv + h) * G * D;
  const int qr_ = (tid & 31) >> 2, qc_ = tid & 3, qks_ = tid >> 5;
  float2 qx0 = make_float2(0.f, 0.f), qx1 = make_float2(0.f, 0.f);
  if (ATT && tid < KS * 32 && qr_ < G) {
    qx0 = __ldcg(reinterpret_cast<const float2*>(qunit + qr_ * D + 16 * qks_ + 2 * qc_));
    qx1 = __ldcg(reinterpret_cast<const float2*>(qunit + qr_ * D + 16 * qks_ + 8 + 2 * qc_));
  }
  bool fits_s = false;
  const int L = call_tokens(Lold_s, a.cap_blocks[s], APPEND, &fits_s);
  const bool app = APPEND && fits_s;
  const int N = ceil_blocks(L);
  const int bpc = (((N + C - 1) / C) + 3) & ~3;
  const int64_t row0 = row_of(a, s, h, 0);
  if (tid <= kPW) mbar_init(bars + tid, 1);
  if (tid == 0) fence_mbar_init();
  if (SEL) {  // hf, xexp, xfine, xref, lh
    uint4* z = reinterpret_cast<uint4*>(hf);
#pragma unroll 1
    for (int i = tid; i < (lay.lh + 256 - lay.hf) / 4; i += kPT) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid < 192) misc[tid] = 0;
  // q as the A operand of S^T = q K^T, split into bf16 high and low parts: lane (r, c) of
  // k-step ks holds head r (zero beyond G) at coordinates 16 ks + 2c, +1 and 16 ks + 8 + 2c, +1
  uint4* qf = reinterpret_cast<uint4*>(psm + lay.qf);
  if (ATT && tid < KS * 32) {  // fragment x = tid (loaded above)
    uint4 v;
    split_bf16(qx0.x * InvSqrtP<D>::v, qx0.y * InvSqrtP<D>::v, v.x, v.z);
    split_bf16(qx1.x * InvSqrtP<D>::v, qx1.y * InvSqrtP<D>::v, v.y, v.w);
    qf[tid] = v;
  }
  __syncthreads();  // misc is zero before warp 0 fills in the plan
  markt(25, 0);
  // the plan, as the stream kernel makes it, from the lengths before this call
  // (no kernel of this call writes seq_len before every post CTA has read it)
  int* sL = reinterpret_cast<int*>(psm + lay.plan);  // [kMaxBatch] tokens of each sequence in this call
  int* sN = sL + kMaxBatch;                           // [kMaxBatch] blocks the stream read
  int* soff = sN + kMaxBatch;
  if (warp == 0) {
    bool f0 = false, f1 = false;
    if (lane < a.B) {
      sL[lane] = call_tokens(sl0, a.cap_blocks[lane], APPEND, &f0);
      sN[lane] = streamed_blocks(sL[lane], APPEND && f0, SEL, a.K, a.scores != nullptr);
    }
    if (lane + 32 < a.B) {
      sL[lane + 32] = call_tokens(sl1, a.cap_blocks[lane + 32], APPEND, &f1);
      sN[lane + 32] = streamed_blocks(sL[lane + 32], APPEND && f1, SEL, a.K, a.scores != nullptr);
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, f0), m1 = __ballot_sync(0xffffffffu, f1);
    if (lane == 0) {
      misc[kMFits] = (int)m0;
      misc[kMFits + 1] = (int)m1;
    }
    __syncwarp();
    plan_warp(sN, a.B, a.Hkv, a.P, stage_blocks(a.r, G), soff, misc + kMPlan, lane);
  }
  __syncthreads();
  markt(26, 0);
  const int seg = misc[kMPlan];
  const int Ns = sN[s];
  const int nseg = (Ns + seg - 1) / seg;
  const int i0 = soff[s] + h * nseg;                 // the unit's first segment record
  const int b_lo = min(N, p * bpc), b_hi = min(N, b_lo + bpc);
  const int nown = b_hi - b_lo;
  const int nown_z = max(0, min(b_hi, Ns) - b_lo);   // of them with zbar / sigma2 from the stream
  const bool all_sel = N <= K;
  const int need0 = K - 3;
  const bool want_keys = SEL && (!all_sel || a.scores);
  const bool hist = SEL && !all_sel && need0 > 0;    // the threshold search runs
  const bool xchg = SEL && !all_sel;                 // the counts are exchanged
  const bool comp = ATT && !(a.variant & kVarNoCompensation) && (!SEL || !all_sel);
  markt(27, 0);

  // ---- a. after the stream: LSE over the records and the open block's a_g (warp 0), zbar and
  // sigma2 rows (warp 1), the compensation share (warps 2..)
  {
    pdl_wait();  // the stream kernel's records, zbar and sigma2 are complete and visible
    if (TRACE && tid == 0) t_wait = global_ns();
    if (warp == 0 && want_keys) {
      const float an = (app && lane < G) ? __ldcg(a.anm + (int64_t)u * G + lane) : -INFINITY;
      record_lse<G>(a, i0, nseg, an, app, lsep, lane);
    }
    markt(22, 0);
    if (warp == 1 && lane == 0 && want_keys && nown_z > 0) {
      const uint32_t bytes = (uint32_t)nown_z * (uint32_t)Gp * 4u;
      mbar_arrive_expect_tx(bars + kPW, 2u * bytes);
      bulk_g2s(zsl, a.zs + (row0 + b_lo) * Gp, bytes, bars + kPW);
      bulk_g2s(ssl, a.ss + (row0 + b_lo) * Gp, bytes, bars + kPW);
      if (!mbar_wait_bounded(bars + kPW, 0u, a.status, s, h, 20)) {
        mbar_drain_bounded(bars + kPW);
        misc[kMBad] = 1;
      }
    }
    markt(23, 32);
    markt(24, 64);
  }
  pdl_trigger();  // the next call's kernels may launch (they wait for this grid before reading)
  __syncthreads();  // LSE parts, a_g of the open block, zsl and ssl in place
  mark(0);

  // ---- b. keys and the local histogram; each thread a run of consecutive blocks
  const int cpt = (nown + kPT - 1) / kPT;
  const int c_lo = min(nown, tid * cpt), c_hi = min(nown, c_lo + cpt);
  if (want_keys) {
    float lse[G];
#pragma unroll
    for (int g = 0; g < G; ++g) lse[g] = lsep[g];
    const bool fom = (a.variant & kVarFirstOrderMass) != 0, nvf = (a.variant & kVarNoVarianceFactor) != 0;
#pragma unroll 1
    for (int i = c_lo; i < c_hi; ++i) {
      const int b = b_lo + i;
      float S = 0.f;
      if (i < nown_z) {  // (the open block, appended in this call, is forced: its S_b is not needed)
        const float lnn = ln_count(b == N - 1 ? L - kBlock * b : kBlock);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float z = zsl[i * Gp + g], s2 = ssl[i * Gp + g];
          const float ph = __expf(lnn + z + (fom ? 0.f : 0.5f * s2) - lse[g]);
          S = fmaf(ph, nvf ? 1.f : s2, S);
        }
      }
      S = fmaxf(S, 0.f);
      const uint32_t key = __float_as_uint(S);
      keys[i] = key;
      if (a.scores) a.scores[(int64_t)u * a.score_stride + b] = S;
      if (hist && b >= 1 && b <= N - 3) atomicAdd(&hf[key >> kDigitShift], 1u);
    }
    __syncthreads();
  }
  mark(1);

  // After barrier 1 every CTA of this cluster has read seq_len (the set-up does); the last
  // cluster to get there writes the lengths after this call's append (a sequence at capacity
  // keeps its own).  One thread of rank 0, off the threshold search's path.
  auto seq_arrive = [&]() {
    if (atomicAdd(a.arrive, 1) == (int)(gridDim.x / C) - 1) {
#pragma unroll 1
      for (int x = 0; x < a.B; ++x) {
        const bool f = ((x < 32 ? misc[kMFits] >> x : misc[kMFits + 1] >> (x - 32)) & 1) != 0;
        if (f) a.seq_len[x] = sL[x];
      }
      a.arrive[0] = 0;
    }
  };

  // ---- the threshold bin T: the histograms summed across the cluster
  uint32_t T = 0xFFFFFFFFu;
  int need = 0;
  bool take_all = true;
  if (hist) {
    uint32_t* h2 = xexp;   // counts per 8-bit key prefix (the exponent)
    uint32_t* h1 = xfine;  // counts per 4-bit key prefix
    {
      // thread e: the 16 fine bins of prefix e
      const int e = tid;  // kPT == 256 prefixes
      const uint4* hv = reinterpret_cast<const uint4*>(hf + e * 16);
      uint32_t ce = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 f = hv[k];
        ce += f.x + f.y + f.z + f.w;
      }
      h2[e] = ce;
      if (ce) atomicAdd(&h1[e >> 4], ce);
    }
    mark(14);
    cluster_sync_all();  // barrier 1: every CTA's histograms are complete (and every CTA has started)
    mark(2);
    if (warp != 0) {
      // the CTA's share of the compensation sums, by the warps idle during the threshold search
      if (comp) comp_share<D, G>(a, i0, nseg, p, C, csh, cR, cW, tid - 32, kPT - 32);
      if (APPEND && p == 0 && tid == 32) seq_arrive();
    } else {
      // three levels of 16 bins over the 12-bit key prefix, each summed over the cluster
      const int3 l1 = cluster_level(h1, C, lane, need0, 0);
      markt(28, 0);
      const int3 l2 = cluster_level(h2 + 16 * l1.x, C, lane, need0, l1.y);
      markt(29, 0);
      const int3 l3 = cluster_level(hf + 16 * (16 * l1.x + l2.x), C, lane, need0, l2.y);
      markt(30, 0);
      if (lane == 0) {
        misc[kMT] = 256 * l1.x + 16 * l2.x + l3.x;
        misc[kMAbove] = l3.y;
        misc[kMCntT] = l3.z;
      }
    }
    __syncthreads();
    T = (uint32_t)misc[kMT];
    need = need0 - misc[kMAbove];
    take_all = misc[kMCntT] == need;
  } else {
    if (comp) comp_share<D, G>(a, i0, nseg, p, C, csh, cR, cW, tid, kPT);
    cluster_sync_all();  // every CTA of the cluster has started before any access to a peer
    if (APPEND && p == 0 && tid == 0) seq_arrive();
  }
  mark(3);

  // ---- c. the sure blocks: forced, above T, or in T when T is taken whole; this CTA's ascending list
  int n_own = 0, ntie = 0;
  if (SEL) {
    auto sure = [&](int i) -> bool {
      const int b = b_lo + i;
      if (all_sel || b == 0 || b >= N - 2) return true;
      if (need0 <= 0) return false;
      const uint32_t bin = keys[i] >> kDigitShift;
      return bin > T || (bin == T && take_all);
    };
    // bitmaps of the sure blocks and of the candidates in bin T (bit i % 32 of word i / 32: block
    // b_lo + i), one ballot per warp and 32 blocks; then warp 0 lists the sure blocks and warp 1 the
    // candidates in ascending order (the rare path's radix areas serve as the bitmaps, and are
    // cleared again afterwards)
    unsigned* sbits = xref;
    unsigned* tbits = xref + 256;
#pragma unroll 1
    for (int i0 = warp * 32; i0 < nown; i0 += kPT) {
      const int i = i0 + lane;
      const bool su = i < nown && sure(i);
      const bool ti = i < nown && !su && !take_all && (keys[i] >> kDigitShift) == T;
      const unsigned sb = __ballot_sync(0xffffffffu, su), tb = __ballot_sync(0xffffffffu, ti);
      if (lane == 0) {
        sbits[i0 >> 5] = sb;
        tbits[i0 >> 5] = tb;
      }
    }
    __syncthreads();
    mark(19);
    const int nwd = (nown + 31) / 32;
    const int cap = nown < K ? nown : K;
    if (warp == 0) {
      const int c = bitmap_list(sbits, nwd, b_lo, own, cap, lane);
      if (lane == 0) misc[kMOwn] = c;
    } else if (warp == 1) {
      // local indices of this CTA's candidates in bin T, and (key, block) of the first kTieCap,
      // read by every CTA of the cluster after barrier 2
      const int c = bitmap_list(tbits, nwd, 0, win, kTieCap, lane);
      if (lane == 0) misc[kMNtie] = c;
      __syncwarp();
      uint2* tiel = reinterpret_cast<uint2*>(xfine + 16);
#pragma unroll 1
      for (int k = lane; k < min(c, kTieCap); k += 32) tiel[k] = make_uint2(keys[win[k]], (uint32_t)(b_lo + win[k]));
    }
    __syncthreads();  // the own list, the candidates and the tie list are complete
    mark(20);
    n_own = min(misc[kMOwn], cap);
    ntie = misc[kMNtie];
#pragma unroll 1
    for (int i = tid; i < 3 * 256; i += kPT) xref[i] = 0u;
  }
  mark(4);
  if (xchg) {
    // this CTA's (own count, tie count), read by every CTA of the cluster after barrier 2
    if (tid == 0) {
      misc[kMMine] = n_own;
      misc[kMMine + 1] = ntie;
    }
    mark(15);
    mark(16);
    cluster_arrive();  // barrier 2 (waited for once this CTA's first copies are in flight)
    mark(17);
  }

  // ---- d, e. attention: this warp's running state
  float am = -INFINITY, al = 0.f;
  float acc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  uint32_t ph = 0u;
  char* stg = reinterpret_cast<char*>(psm + lay.stg);
  stg += (1024u - (smem_u32(stg) & 1023u)) & 1023u;  // the swizzled boxes want 1024-byte alignment
  stg += warp * stg_bytes(D);
  const int* selrow_in = a.sel + (int64_t)u * K;
  int tot_sel = 0;
  if (ATT && !SEL) {
    // the caller's selection: entries that are not ascending or not inside [0, N) are skipped and reported
    int bad = 0, cntv = 0;
#pragma unroll 1
    for (int i = tid; i < K; i += kPT) {
      const int e = __ldcg(selrow_in + i);
      const int prev = i > 0 ? __ldcg(selrow_in + i - 1) : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      cntv += ok;
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cntv = __reduce_add_sync(0xffffffffu, cntv);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cntv) atomicAdd(misc + kMTot, cntv);
      if (bad) misc[kMBad] |= 2;
    }
    __syncthreads();
    tot_sel = misc[kMTot];
    if ((misc[kMBad] & 2) && p == 0 && tid == 0) set_error(a.status, kDevBadSelection, s, h, 61);
  }
  const bool comp_blk = comp && (SEL || tot_sel < N);
  auto n_of = [&](int b) { return (b == N - 1) ? L - kBlock * b : kBlock; };
  // compensation of block b comes off unless this call appended it (the stream skipped it then)
  auto comp_of = [&](int b) { return comp_blk && !(APPEND && app && b == N - 1); };
  // stage block b into this warp's buffer: its 16 K and 16 V rows by 2 D / 64 tensor copies (the
  // rows past a partial block's tokens are zeroed once they land); returns zbar of head lane / 4
  bool dirty = false;  // this warp zeroed rows of its buffer with ordinary stores
  auto issue = [&](int b) -> float {
    const int64_t row = row0 + b;
    const bool cb = comp_of(b);
    __syncwarp();  // the buffer's previous contents are read
    const bool plain = a.kv_host || !a.tmap_ok;
    if (plain) {
      // K and V in host memory (or no tensor maps): every lane copies 16-byte chunks of the block's n rows into their
      // swizzled places (rows past n are masked for K and zeroed for V once the copies land)
      plain_copy<D>(stg, reinterpret_cast<const char*>(a.k + row * kBlock * D),
                    reinterpret_cast<const char*>(a.v + row * kBlock * D), n_of(b), lane);
    }
    if (lane == 0) {
      // ordinary stores into the buffer are ordered before the copies that overwrite it
      if (dirty) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(bars + warp, (plain ? 0u : 2u * (uint32_t)stg_kv(D)) + (cb ? D * 4u : 0u));
      if (!plain) {
        const int y = (int)((a.layer_row0 + row) * kBlock);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          tma_2d(stg + hh * kBlock * 128, a.tmap_k, 64 * hh, y, bars + warp, pol);
          tma_2d(stg + stg_kv(D) + hh * kBlock * 128, a.tmap_v, 64 * hh, y, bars + warp, pol);
        }
      }
      if (cb) bulk_g2s_hint(stg + 2 * stg_kv(D), a.vbar + row * D, D * 4u, bars + warp, pol);
    }
    dirty = false;
    return (cb && (lane >> 2) < G) ? __ldcg(a.zs + row * Gp + (lane >> 2)) : 0.f;
  };
  // after the copies of block b landed: V rows past its tokens hold whatever follows them in the
  // cache; zero them (whole rows, so the swizzle does not matter)
  auto clear_tail = [&](int n) {
    if (n < kBlock) {
      for (int x = lane; x < (kBlock - n) * (D / 8); x += 32) {
        const int t = n + x / (D / 8), j = x % (D / 8);
        *reinterpret_cast<uint4*>(stg + stg_kv(D) + (j >> 3) * kBlock * 128 + t * 128 + (j & 7) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      dirty = true;
      __syncwarp();
    }
  };

  // this CTA's own sure blocks from the top of its list (the open block, the last, comes first):
  // their copies start before the exchange settles
  const int mine0 = min(n_own, kPW);
  int b_cur = -1;
  float zb_cur = 0.f;
  if (ATT && SEL) {
    b_cur = warp < n_own ? own[n_own - 1 - warp] : -1;
    if (xchg) misc[kMR0 + warp] = b_cur;
    if (b_cur >= 0) zb_cur = issue(b_cur);
    mark(18);
  }
  mark(5);

  // ---- d. after the exchange: the tie winners and the rest of the work
  int own_base = b_lo;  // this CTA's offset in the ascending selection
  int nwin = 0;
  bool rare = false;
  int OV = 0, SP = 0, spx_p = 0, total = 0, ov = 0, ovx = 0;  // work items of the common path
  if (xchg) {
    cluster_wait();  // barrier 2: every count and tie list is here
    mark(6);
    // every warp alike: lane q < C holds CTA q's counts
    const uint2 cq = lane < C ? ld_peer_u2(peer_smem(misc + kMMine, (uint32_t)lane)) : make_uint2(0u, 0u);
    const int co = (int)cq.x, ct = (int)cq.y;
    ov = max(0, co - kPW);
    const int sp = lane < C ? kPW - min(co, kPW) : 0;
    int io = co, it = ct, iv = ov, is = sp, mx = ct;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, io, o), y1 = __shfl_up_sync(0xffffffffu, it, o);
      const int y2 = __shfl_up_sync(0xffffffffu, iv, o), y3 = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        io += y0;
        it += y1;
        iv += y2;
        is += y3;
      }
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const int sum_own = __shfl_sync(0xffffffffu, io, 31), nt_all = __shfl_sync(0xffffffffu, it, 31);
    OV = __shfl_sync(0xffffffffu, iv, 31);
    SP = __shfl_sync(0xffffffffu, is, 31);
    ovx = iv - ov;                                   // lane q: first overflow item of CTA q
    spx_p = __shfl_sync(0xffffffffu, is - sp, p);    // first idle slot of this CTA
    const int opre_p = __shfl_sync(0xffffffffu, io - co, p);
    rare = !take_all && need > 0 && (mx > kTieCap || nt_all > kRankMax);
    if (!rare) {
      if (!take_all && need > 0) {
        // rank every tie entry among all (key desc, block asc), one warp per entry over a
        // dense copy of the lists; the first `need` win, kept in rank order
        if (warp == 0 && lane < C) {
          misc[kMTpre + lane] = it - ct;
          misc[kMTcnt + lane] = ct;
        }
        __syncthreads();
        const uint2* tiel = reinterpret_cast<const uint2*>(xfine + 16);
        static_assert(kMaxC * kTieCap == 4 * kPT, "four tie entries per thread");
        uint2 tv[4];
        int td[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // every load first, then the stores
          const int e = tid + j * kPT, q = e / kTieCap, k = e % kTieCap;
          const bool ok = q < C && k < misc[kMTcnt + q];
          td[j] = ok ? misc[kMTpre + q] + k : -1;
          tv[j] = ok ? ld_peer_u2(peer_smem(tiel + k, (uint32_t)q)) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (td[j] >= 0) dense[td[j]] = tv[j];
        __syncthreads();
        // entry j by a group of tpe consecutive threads (the most that fit, up to a warp), which
        // split the comparisons; its rank is the count of entries ahead of it
        int tpe = 1;
        while (tpe < 32 && nt_all * 2 * tpe <= kPT) tpe <<= 1;
        const int j = tid / tpe, part = tid % tpe;
        const bool live = j < nt_all;
        const uint2 me = live ? dense[j] : make_uint2(0u, 0u);
        int rank = 0;
        if (live) {
#pragma unroll 4
          for (int j2 = part; j2 < nt_all; j2 += tpe) {
            const uint2 o = dense[j2];
            rank += (o.x > me.x) || (o.x == me.x && o.y < me.y);
          }
        }
#pragma unroll 1
        for (int o = 1; o < tpe; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (live && part == 0 && rank < need) win[rank] = (int)me.y;
        nwin = need;
        __syncthreads();
      }
      mark(7);
      tot_sel = sum_own + nwin;
      total = OV + nwin;
      // this CTA's offset in the ascending selection: the lists of the lower ranks and the
      // tie winners below this CTA's blocks
      int below = 0;
#pragma unroll 1
      for (int k = lane; k < nwin; k += 32) below += win[k] < b_lo;
      own_base = opre_p + __reduce_add_sync(0xffffffffu, below);
    } else {
      // rare: resolve bin T by more radix digits; every CTA attends its own winners itself
      const int3 rr = rare_select(keys, reinterpret_cast<unsigned*>(dense), own, n_own, nown, b_lo, N, K, T, need,
                                  xref, lh, misc, C, p);
      n_own = rr.x;
      own_base = rr.y;
      tot_sel = rr.z;
      mark(7);
    }
  } else if (SEL) {
    tot_sel = N;
    own_base = b_lo;
  }
  mark(8);

  // the next block of this warp's work, round `rd` (-1: none left, -2: skip this round)
  auto next_block = [&](int rd) -> int {
    if (!SEL) {  // the caller's selection, spread over the cluster's warps round by round
      const int j = (rd * C + p) * kPW + warp;
      if (j >= K) return -1;
      const int e = __ldcg(selrow_in + j);
      const int prev = j > 0 ? __ldcg(selrow_in + j - 1) : -1;
      return (e >= 0 && e < N && (j == 0 || (prev >= 0 && prev < e))) ? e : -2;
    }
    if (all_sel) {  // every block: this CTA's own list from the top, kPW per round
      const int k = n_own - 1 - warp - kPW * rd;
      return k >= 0 ? own[k] : -1;
    }
    if (rare) {  // this CTA's final list, minus the blocks started before the exchange
      const int k = warp + kPW * rd;
      if (k >= n_own) return -1;
      const int b = own[k];
#pragma unroll 1
      for (int w = 0; w < kPW; ++w)
        if (misc[kMR0 + w] == b) return -2;
      return b;
    }
    // items: the own lists beyond their top kPW (CTA by CTA), then the tie winners; slots:
    // the warps idle before the exchange (CTA by CTA), then every warp round by round
    const int k = rd == 0 ? spx_p + warp - mine0 : SP + ((rd - 1) * C + p) * kPW + warp;
    if (k >= total) return -1;
    if (k < OV) {
      const unsigned bal = __ballot_sync(0xffffffffu, lane < C && ov > 0 && ovx <= k);
      const int q = 31 - __clz(bal);
      return (int)ld_peer_u32(peer_smem(own + (k - __shfl_sync(0xffffffffu, ovx, q)), (uint32_t)q));
    }
    return win[k - OV];
  };
  // warps without a block in flight start their first one now; the selection is written while
  // the copies land
  int rd = (SEL && !rare && warp < mine0) ? 1 : 0;
  auto fetch = [&]() -> bool {
    int nb = -2;
#pragma unroll 1
    while (nb == -2) nb = next_block(rd++);
    if (nb < 0) return false;
    b_cur = nb;
    zb_cur = issue(nb);
    return true;
  };
  bool have = b_cur >= 0;
  if (ATT && !have) have = fetch();
  if (SEL) {
    // the ascending selection from own_base on: this CTA's sure blocks, and the tie winners among
    // its blocks
    int* selrow = a.sel + (int64_t)u * K;
    if (nwin > 0) {
      // both as one bitmap of the CTA's blocks (in the fine histogram's place, which no peer
      // reads after barrier 2), listed in ascending order by warp 0
      if (warp == 0) {
        unsigned* bits = hf;
        const int nwd = (nown + 31) / 32;
#pragma unroll 1
        for (int w = lane; w < nwd; w += 32) bits[w] = 0u;
        __syncwarp();
#pragma unroll 1
        for (int e = lane; e < n_own; e += 32) atomicOr(&bits[(own[e] - b_lo) >> 5], 1u << ((own[e] - b_lo) & 31));
#pragma unroll 1
        for (int k = lane; k < nwin; k += 32) {
          const int b = win[k];
          if (b >= b_lo && b < b_hi) atomicOr(&bits[(b - b_lo) >> 5], 1u << ((b - b_lo) & 31));
        }
        __syncwarp();
        bitmap_list(bits, nwd, b_lo, selrow + own_base, K - own_base, lane);
      }
    } else {
#pragma unroll 1
      for (int e = tid; e < n_own; e += kPT)
        if (own_base + e < K) selrow[own_base + e] = own[e];
    }
    if (p == 0) {
#pragma unroll 1
      for (int i = tot_sel + tid; i < K; i += kPT) selrow[i] = -1;
      if (tid == 0 && tot_sel != (N < K ? N : K)) set_error(a.status, kDevInternal, s, h, 50);
    }
  }
  mark(9);
  if (ATT) {
    // one attention site: the block whose copy is in flight, then the next
#pragma unroll 1
    while (have) {
      if (!mbar_wait_bounded(bars + warp, ph, a.status, s, h, 62)) {
        mbar_drain_bounded(bars + warp);
        misc[kMBad] |= 1;
        break;
      }
      ph ^= 1u;
      if (a.kv_host || !a.tmap_ok) {  // this lane's copies, then every lane's
        cp_async_wait_all();
        __syncwarp();
      }
      clear_tail(n_of(b_cur));
      blk_attend<D, G>(am, al, acc, qf, stg, n_of(b_cur), comp_of(b_cur), zb_cur, lane);
      if (misc[kMBad] & 1) break;
      have = fetch();
    }
  }
  const unsigned long long t_sel = TRACE ? global_ns() : 0ull;
  if (SEL && !ATT) {
    // score/select only: no peer reads this CTA's shared memory after the barrier
    cluster_sync_all();
    if (TRACE && tid == 0 && a.Q + a.P + (int)blockIdx.x < a.trace_cap) {
      unsigned long long* rr = a.trace + 1 + 8 * (int64_t)(a.Q + a.P + blockIdx.x);
      rr[0] = ((unsigned long long)blockIdx.x << 32) | (1ull << 24) | (unsigned)p;
      rr[1] = (unsigned long long)u; rr[2] = t_start; rr[3] = t_wait; rr[4] = t_sel; rr[5] = t_sel;
    }
    return;
  }
  const unsigned long long t_att = t_sel;

  // ---- the CTA's partial: its warps and its compensation share
  markt(31, 0);
  __syncthreads();  // the staging is free: the partials reuse the union
  markt(32, 0);
  float* red_a = psm + lay.red;            // [kPW][8][D]
  float* red_m = red_a + kPW * D * 8;      // [kPW][8]
  float* red_l = red_m + kPW * 8;          // [kPW][8]
  {
    const int r = lane >> 2, c = lane & 3;
    if (c == 0 && r < G) {
      red_m[warp * 8 + r] = am;
      red_l[warp * 8 + r] = al;
    }
    float* ra = red_a + (warp * 8 + 2 * c) * D + r;  // head 2c; head 2c + 1 is D further
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      if (2 * c < G) {
        ra[16 * mt] = acc[mt][0];
        ra[16 * mt + 8] = acc[mt][2];
      }
      if (2 * c + 1 < G) {
        ra[D + 16 * mt] = acc[mt][1];
        ra[D + 16 * mt + 8] = acc[mt][3];
      }
    }
  }
  __syncthreads();
  mark(10);
  // per float4 column item: the warps' parts (and the share) at their common maximum, pushed to
  // the rank that merges the item
  const int items = G * D / 4;
  const int ipr = post_ipr(D, G, C);
#pragma unroll 1
  for (int i4 = tid; i4 < items; i4 += kPT) {
    const int g = (4 * i4) / D, col = (4 * i4) % D;
    float M = comp_blk ? cR[g] : -INFINITY;
#pragma unroll
    for (int w = 0; w < kPW; ++w) M = fmaxf(M, red_m[w * 8 + g]);
    float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kPW; ++w) {
        const float mw = red_m[w * 8 + g];
        const float f = mw == -INFINITY ? 0.f : __expf(mw - M);
        Ls = fmaf(f, red_l[w * 8 + g], Ls);
        const float4 x = *reinterpret_cast<const float4*>(red_a + (w * 8 + g) * D + col);
        as.x = fmaf(x.x, f, as.x);
        as.y = fmaf(x.y, f, as.y);
        as.z = fmaf(x.z, f, as.z);
        as.w = fmaf(x.w, f, as.w);
      }
      if (comp_blk && cR[g] != -INFINITY) {
        const float f = __expf(cR[g] - M);
        const float4 x = *reinterpret_cast<const float4*>(csh + g * D + col);
        Ls = fmaf(f, cW[g], Ls);
        as.x = fmaf(x.x, f, as.x);
        as.y = fmaf(x.y, f, as.y);
        as.z = fmaf(x.z, f, as.z);
        as.w = fmaf(x.w, f, as.w);
      }
    }
    const int rk = i4 / ipr, il = i4 - rk * ipr;
    const uint32_t dst = peer_smem(xm + (il * C + p) * 8, (uint32_t)rk);
    st_peer_f4(dst, as);
    st_peer_u2(dst + 16u, make_uint2(__float_as_uint(M), __float_as_uint(Ls)));
  }
  mark(11);
  cluster_sync_all();  // barrier 3: every partial of this rank's columns is here; no CTA touches a peer after this
  mark(12);
  // this rank's column items: Cp (C rounded up to a power of two) lanes per item, lane q
  // takes CTA q's partial; the partials are merged across those lanes
  {
    const int i_lo = p * ipr, i_hi = min(items, i_lo + ipr);
    int Cp = 1;
    while (Cp < C) Cp <<= 1;
    const int nx = max(0, i_hi - i_lo) * Cp;  // groups of Cp lanes never straddle a warp (Cp divides 32)
#pragma unroll 1
    for (int x0 = warp * 32; x0 < nx; x0 += kPT) {
      const int x = x0 + lane;
      const bool live = x < nx;
      const int il = x / Cp, q = x % Cp;
      const int i4 = i_lo + il, g = (4 * i4) / D, col = (4 * i4) % D;
      float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
      float mq = -INFINITY, lq = 0.f;
      if (live && q < C) {
        const float* e = xm + (il * C + q) * 8;
        as = *reinterpret_cast<const float4*>(e);
        mq = e[4];
        lq = e[5];
      }
      float M = mq;
#pragma unroll 1
      for (int o = 1; o < Cp; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = (M == -INFINITY || mq == -INFINITY) ? 0.f : __expf(mq - M);
      as.x *= f;
      as.y *= f;
      as.z *= f;
      as.w *= f;
      lq *= f;
#pragma unroll 1
      for (int o = 1; o < Cp; o <<= 1) {
        as.x += __shfl_xor_sync(0xffffffffu, as.x, o);
        as.y += __shfl_xor_sync(0xffffffffu, as.y, o);
        as.z += __shfl_xor_sync(0xffffffffu, as.z, o);
        as.w += __shfl_xor_sync(0xffffffffu, as.w, o);
        lq += __shfl_xor_sync(0xffffffffu, lq, o);
      }
      if (live && q == 0) {
        const float inv = lq > 0.f ? 1.f / lq : 0.f;
        float* out = a.out + ((int64_t)s * a.Hkv + h) * G * D;
        *reinterpret_cast<float4*>(out + g * D + col) = make_float4(as.x * inv, as.y * inv, as.z * inv, as.w * inv);
      }
    }
  }
  mark(13);
  if (TRACE && tid == 0) {
    for (int rec = 0; rec < 5; ++rec) {
      const int64_t ri = a.Q + a.P + (int64_t)(1 + rec) * gridDim.x + blockIdx.x;
      if (ri < a.trace_cap) {
        a.trace[1 + 8 * ri] = ((unsigned long long)blockIdx.x << 32) | ((2ull + rec) << 24) |
                              (unsigned)(ntie | (n_own << 12));
        for (int k = 0; k < 7; ++k) a.trace[1 + 8 * ri + 1 + k] = 7 * rec + k < 35 ? tmk[7 * rec + k] : 0ull;
      }
    }
    if (a.Q + a.P + (int)blockIdx.x < a.trace_cap) {
      unsigned long long* rr = a.trace + 1 + 8 * (int64_t)(a.Q + a.P + blockIdx.x);
      rr[0] = ((unsigned long long)blockIdx.x << 32) | (1ull << 24) | (unsigned)p;
      rr[1] = (unsigned long long)u;
      rr[2] = t_start;
      rr[3] = t_wait;
      rr[4] = t_sel;
      rr[5] = t_att;
      rr[6] = global_ns();
      rr[7] = (unsigned long long)tot_sel;
    }
  }
}

template <int D, int G, int MODE>
static cudaError_t launch_post_mode(const LayerArgs& a, cudaStream_t st) {
  const void* fn = a.trace ? reinterpret_cast<const void*>(&k_post<D, G, MODE, true>)
                           : reinterpret_cast<const void*>(&k_post<D, G, MODE, false>);
  // (shared memory limit and cluster size allowed by prepare_post)
  const size_t smem = (size_t)post_layout(D, G, a.C, a.bpc_max, a.K).total * 4;
  LayerArgs args = a;
  chain_split(args, MODE);
  void* argv[] = {&args};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.Hkv * a.C));
  cfg.blockDim = dim3(kPT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)a.C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelExC(&cfg, fn, argv);
}

template <int D, int G>
static cudaError_t launch_post_dg(const LayerArgs& a, int mode, cudaStream_t st) {
  switch (mode) {
    case kFusedDecode: return launch_post_mode<D, G, kFusedDecode>(a, st);
    case kFusedScoreSelect: return launch_post_mode<D, G, kFusedScoreSelect>(a, st);
    case kFusedAttend: return launch_post_mode<D, G, kFusedAttend>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_post(const LayerArgs& a, int mode, cudaStream_t st) {
#define COMPKV_G(DD)                                       \
  switch (a.G) {                                           \
    case 1: return launch_post_dg<DD, 1>(a, mode, st);     \
    case 2: return launch_post_dg<DD, 2>(a, mode, st);     \
    case 4: return launch_post_dg<DD, 4>(a, mode, st);     \
    case 8: return launch_post_dg<DD, 8>(a, mode, st);     \
    default: return cudaErrorInvalidValue;                 \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

size_t post_smem(int D, int G, int C, int bpc_max, int K) { return (size_t)post_layout(D, G, C, bpc_max, K).total * 4; }

template <int D, int G, int MODE>
static cudaError_t prepare_post_mode(int C, int bpc_max, int K) {
  cudaError_t e = cudaSuccess;
  for (const void* fn : {reinterpret_cast<const void*>(&k_post<D, G, MODE, false>),
                         reinterpret_cast<const void*>(&k_post<D, G, MODE, true>)}) {
    if (e == cudaSuccess) e = raise_smem_limit(fn, post_layout(D, G, C, bpc_max, K).total * 4);
    if (e == cudaSuccess && C > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  }
  return e;
}

template <int D, int G>
static cudaError_t prepare_post_dg(int C, int bpc_max, int K) {
  cudaError_t e = prepare_post_mode<D, G, kFusedDecode>(C, bpc_max, K);
  if (e == cudaSuccess) e = prepare_post_mode<D, G, kFusedScoreSelect>(C, bpc_max, K);
  if (e == cudaSuccess) e = prepare_post_mode<D, G, kFusedAttend>(C, bpc_max, K);
  return e;
}

cudaError_t prepare_post(int D, int G, int C, int bpc_max, int K) {
#define COMPKV_G(DD)                                        \
  switch (G) {                                              \
    case 1: return prepare_post_dg<DD, 1>(C, bpc_max, K);   \
    case 2: return prepare_post_dg<DD, 2>(C, bpc_max, K);   \
    case 4: return prepare_post_dg<DD, 4>(C, bpc_max, K);   \
    case 8: return prepare_post_dg<DD, 8>(C, bpc_max, K);   \
    default: return cudaErrorInvalidValue;                  \
  }
  if (D == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

}  // namespace compkv
