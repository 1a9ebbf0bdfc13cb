// Selection, exact attention and Mean compensation of the CompKV decode step
// (onedev.kr/papers/157), after the summary stream (stream_kernel.cu).
//
// One thread-block cluster of C CTAs per (sequence, KV head) unit.  CTA rank p
// owns the unit's blocks [p bpc, (p + 1) bpc) (bpc = ceil(N / C) rounded up
// to 4) and, of the stream's segment records, those with index = p (mod C):
//   a. LSE_g = logsumexp_b a_{g,b} from all segment records (each CTA alone);
//      S_b = sum_g phat_{g,b} sigma2_{g,b} ("무엇과 다른가") of its blocks as
//      order-preserving keys, and their 12-bit histogram (candidates 1..N-3);
//   b. the histograms summed across the cluster in distributed shared memory
//      (exponent bins at rank 0, the 16 fine bins of exponent e at rank e % C);
//      every CTA finds the threshold bin T where the count of larger keys
//      reaches K - 3 (the forced sink block and the two most recent blocks
//      take the other three places of the budget);
//   c. every CTA classifies its own blocks and pushes, in one exchange, its
//      count of selected blocks and the keys of its blocks in T when T must be
//      ranked (ties to the lower block index); every CTA ranks those few keys
//      itself, so after one cluster barrier all CTAs know the whole selection;
//   d. the selected blocks are spread over the cluster's warps (one block per
//      warp and round); each warp attends exactly to its block's bf16 K/V and
//      removes the block's own Mean-compensation term, which the stream added
//      for every block ("어떻게 동작하나": unselected blocks contribute
//      |b| e^{zbar} vbar and |b| e^{zbar}); the partials, with the CTA's share
//      of the compensation sums, merge across the cluster into out = acc / l.
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

// Shared memory of the post kernel, in 4-byte words.
struct PostLayout {
  int zsl, ssl, keys, own, bits, csh, plan, U, hf, he, xexp, xfine, xref, lh, tie, stg, stg_w, red, xm, misc, win, bars, total;
};
__host__ __device__ inline int post_items(int D, int G) { return G * D / 4; }
__host__ __device__ inline int post_ipr(int D, int G, int C) { return (post_items(D, G) + C - 1) / C; }
__host__ __device__ inline PostLayout post_layout(int D, int G, int C, int bpc_max, int K) {
  PostLayout l;
  const int Gp = pad_g(G);
  int o = 0;
  l.zsl = o; o += bpc_max * Gp;
  l.ssl = o; o += bpc_max * Gp;
  l.keys = o; o += (bpc_max + 3) & ~3;
  l.own = o; o += ((bpc_max < K ? bpc_max : K) + 7) & ~3;
  l.bits = o; o += (bpc_max + 31) / 32 + 4;
  o = (o + 3) & ~3;
  l.csh = o; o += G * D;           // this CTA's share of the compensation numerator [G][D]
  l.plan = o; o += 3 * kMaxBatch + 4;  // tokens, blocks and first segment of every sequence
  // union: selection (local histograms | exchanged histograms | tie lists) / attention staging / CTA partials
  l.U = o;
  l.hf = o;                        // local 12-bit histogram [4096]; later the tie lists [C][kTieCap] x (key, index)
  l.tie = o;
  l.he = l.hf + kFine;             // local exponent histogram [256]
  l.xexp = l.he + 256;             // exchanged exponent histogram (rank 0) [256]
  l.xfine = l.xexp + 256;          // exchanged fine bins of this rank's exponents [ceil(256 / C) * 16]
  l.xref = l.xfine + ((256 + C - 1) / C) * 16;  // refinement histograms (rank 0) [3][256]
  l.lh = l.xref + 3 * 256;         // refinement local histogram [256]
  const int selw = l.lh + 256 - o;
  l.stg = o;                       // attention: per warp K, V rows (bf16) and z, p [kBlock][G]
  l.stg_w = kBlock * D + 2 * kBlock * G;
  const int attw = kPW * l.stg_w;
  const int redw = kPW * G * D + 2 * kPW * G + G * (kPW + 1) + 2 * G;
  l.red = o;                       // CTA partials after the attention: [kPW][G][D], m, l [kPW][G]
  int uw = selw > attw ? selw : attw;
  uw = uw > redw ? uw : redw;
  o += (uw + 3) & ~3;
  l.xm = o; o += post_ipr(D, G, C) * C * 8;   // merge staging: [items per rank][C][acc4, m, l, -, -]
  l.win = o; o += kRankMax + 4;               // tie winners in rank order
  l.misc = o; o += 192;
  l.bars = o; o += 2 * (kPW + 2);
  l.total = o;
  return l;
}

// misc slots (ints unless noted)
enum : int {
  kMT = 0, kMAbove, kMCntT, kMNtie, kMOwn, kMTake, kMNeed, kMBad, kMNwin, kMTot,
  kMLse = 16,        // float [8]
  kMCR = 24,         // float [8]: compensation reference of this CTA's share
  kMCW = 32,         // float [8]: compensation weight sum of the share
  kMCnt = 40,        // int2 [16]: per CTA (own selected count, tie count), pushed by the peers
  kMCntR = 72,       // int [16]: refinement counts, pushed by the peers
  kMScan = 88,       // int [8]: scan scratch
  kMPlan = 96,       // seg, total
  kMFits = 100,      // [2] bit s: sequence s had room for its token
  kMSumOwn = 102, kMNtAll, kMMx, kMWBelow,
  kMOpre = 112,      // [17] exclusive prefix of the CTAs' own-list counts
  kMTpre = 132,      // [17] exclusive prefix of the CTAs' tie counts
};

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
#pragma unroll
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
__device__ __forceinline__ int bitmap_list(const unsigned* words, int nw, int lo, int* list, int cap, int lane) {
  const int per = (nw + 31) / 32;
  int loc = 0;
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

// Rare path of the selection: more keys share the threshold bin T than the
// tie lists hold.  The keys in play (own candidates in bin T) are resolved by
// three more radix digits (bits 18..11, 10..3, 2..0), each a histogram summed
// at rank 0 with one cluster barrier, and keys equal in every bit go to the
// lowest block indices (counts exchanged, one more barrier).  Sets the bits of
// the selected in-play blocks in `bits`.  Called by every thread of every CTA
// of the cluster.
__device__ __noinline__ void refine_select(const uint32_t* keys, unsigned* bits, int nown, int b_lo, int N, uint32_t T,
                                           int need, uint32_t* xref, uint32_t* lh, int* misc, int C, int p) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t pfx = T << kDigitShift, pm = 0xFFFFFFFFu << kDigitShift;
  bool done = false;
  for (int level = 1; level <= 3 && !done; ++level) {
    const int shift = level == 1 ? 11 : (level == 2 ? 3 : 0);
    const int nb = level == 3 ? 8 : 256;
    const uint32_t dm = (uint32_t)nb - 1u;
    for (int i = tid; i < 256; i += kPT) lh[i] = 0u;
    __syncthreads();
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      if (b < 1 || b > N - 3) continue;
      const uint32_t key = keys[i];
      if ((key & pm) == pfx && !((bits[i >> 5] >> (i & 31)) & 1u)) atomicAdd(&lh[(key >> shift) & dm], 1u);
    }
    __syncthreads();
    uint32_t* xr = xref + (level - 1) * 256;
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
    for (int q = 0; q < p; ++q) before += misc[kMCntR + q];
    int take = need - before;
    take = take < 0 ? 0 : (take > tot ? tot : take);
    if (warp == 0 && take > 0) {
      // the first `take` in-play blocks in index order: one lane scans
      if (lane == 0) {
        int got = 0;
        for (int i = 0; i < nown && got < take; ++i) {
          const int b = b_lo + i;
          if (b < 1 || b > N - 3) continue;
          if ((keys[i] & pm) == pfx && !((bits[i >> 5] >> (i & 31)) & 1u)) {
            bits[i >> 5] |= 1u << (i & 31);
            ++got;
          }
        }
      }
    }
    __syncthreads();
  }
}

template <int D, int G, int MODE>
__global__ void __launch_bounds__(kPT, 2) k_post(LayerArgs a) {
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool ATT = (MODE & kFAttend) != 0;
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr int V = D / 32;                                          // coordinates per lane
  constexpr int TG = G >= 8 ? 2 : ((32 / G) > 16 ? 16 : (32 / G));  // tokens per reduction group
  constexpr int P = TG * G;                                          // values per group (16 or 32)
  constexpr int W = V / 2;                                           // 32-bit words of a token slice
  constexpr int NG = kBlock / TG;
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
  unsigned* bits = reinterpret_cast<unsigned*>(psm + lay.bits);
  uint32_t* hf = reinterpret_cast<uint32_t*>(psm + lay.hf);
  uint32_t* he = reinterpret_cast<uint32_t*>(psm + lay.he);
  uint32_t* xexp = reinterpret_cast<uint32_t*>(psm + lay.xexp);
  uint32_t* xfine = reinterpret_cast<uint32_t*>(psm + lay.xfine);
  uint32_t* xref = reinterpret_cast<uint32_t*>(psm + lay.xref);
  uint32_t* lh = reinterpret_cast<uint32_t*>(psm + lay.lh);
  uint2* tie = reinterpret_cast<uint2*>(psm + lay.tie);   // [C][kTieCap] (key, block), after the histograms
  float* xm = psm + lay.xm;
  int* win = reinterpret_cast<int*>(psm + lay.win);
  int* misc = reinterpret_cast<int*>(psm + lay.misc);
  float* lse = reinterpret_cast<float*>(misc + kMLse);
  float* cR = reinterpret_cast<float*>(misc + kMCR);
  float* cW = reinterpret_cast<float*>(misc + kMCW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(psm + lay.bars);  // [kPW] attention, [kPW] = zbar/sigma2 load
  const unsigned long long t_start = a.trace ? global_ns() : 0ull;
  unsigned long long pmk[7] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
  auto mark = [&](int k) {
    if (a.trace) pmk[k] = global_ns();
  };

  // ---- set-up before the stream's results are visible
  if (tid <= kPW) mbar_init(bars + tid, 1);
  fence_mbar_init();
  if (SEL) {
    for (int i = tid; i < 256 + ((256 + C - 1) / C) * 16 + 3 * 256; i += kPT) xexp[i] = 0u;  // (xexp,) xfine, xref
  }
  if (tid < 192) misc[tid] = 0;
  float qr[G][V];
  if (ATT) {
    const float* qg = a.q + ((int64_t)s * a.Hkv + h) * G * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < V; ++i) qr[g][i] = qg[g * D + lane * V + i] * InvSqrtP<D>::v;
  }
  __syncthreads();  // misc is zero before warp 0 fills in the plan
  // the plan, as the stream kernel makes it, from the lengths before this call
  // (no kernel of this call writes seq_len before every post CTA has read it)
  int* sL = reinterpret_cast<int*>(psm + lay.plan);  // [kMaxBatch] tokens of each sequence in this call
  int* sN = sL + kMaxBatch;
  int* soff = sN + kMaxBatch;
  if (warp == 0) {
    bool f0 = false, f1 = false;
    if (lane < a.B) sL[lane] = call_tokens(__ldcg(a.seq_len + lane), a.cap_blocks[lane], APPEND, &f0);
    if (lane + 32 < a.B) sL[lane + 32] = call_tokens(__ldcg(a.seq_len + lane + 32), a.cap_blocks[lane + 32], APPEND, &f1);
    const unsigned m0 = __ballot_sync(0xffffffffu, f0), m1 = __ballot_sync(0xffffffffu, f1);
    if (lane == 0) {
      misc[kMFits] = (int)m0;
      misc[kMFits + 1] = (int)m1;
    }
    __syncwarp();
    plan_warp(sL, a.B, a.Hkv, a.P, stage_blocks(a.r, G), sN, soff, misc + kMPlan, lane);
  }
  __syncthreads();
  const int seg = misc[kMPlan];
  const int L = sL[s], N = sN[s];
  const int nseg = (N + seg - 1) / seg;
  const int i0 = soff[s] + h * nseg;                 // the unit's first segment record
  const int bpc = (((N + C - 1) / C) + 3) & ~3;
  const int b_lo = min(N, p * bpc), b_hi = min(N, b_lo + bpc);
  const int nown = b_hi - b_lo;
  const int64_t row0 = row_of(a, s, h, 0);
  const bool all_sel = N <= K;
  const bool comp_on = !(a.variant & kVarNoCompensation);
  const bool want_keys = SEL && (!all_sel || a.scores);
  cluster_arrive();  // this CTA's exchange histograms are zero (waited for before the first push)
  pdl_wait();        // the stream kernel's records, zbar and sigma2 are complete and visible
  pdl_trigger();     // the next call's kernels may launch (they wait for this grid before reading)
  const unsigned long long t_wait = a.trace ? global_ns() : 0ull;

  // zbar (and sigma2) of this CTA's blocks into shared memory
  if (tid == 0 && nown > 0 && (want_keys || ATT)) {
    const uint32_t bytes = (uint32_t)nown * (uint32_t)Gp * 4u;
    mbar_arrive_expect_tx(bars + kPW, want_keys ? 2u * bytes : bytes);
    bulk_g2s(zsl, a.zs + (row0 + b_lo) * Gp, bytes, bars + kPW);
    if (want_keys) bulk_g2s(ssl, a.ss + (row0 + b_lo) * Gp, bytes, bars + kPW);
  }
  // LSE_g over all blocks from the unit's segment records (warp g)
  if (want_keys && warp < G) {
    const int g = warp;
    float M = -INFINITY, S = 0.f;
#pragma unroll 1
    for (int k0 = 0; k0 < nseg; k0 += 128) {  // four records per lane in flight at once
      float4 e[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + lane + 32 * j;
        e[j] = k < nseg ? __ldcg(a.rec + (int64_t)(i0 + k) * G + g) : make_float4(-INFINITY, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) lse_merge(M, S, e[j].x, e[j].y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      lse_merge(M, S, M2, S2);
    }
    if (lane == 0) lse[g] = M + logf(S);
  }
  // this CTA's share of the compensation sums: segment records p, p + C, ...
  // rescaled to their common maximum; thread items (head, column quad), every
  // load issued before any is used
  const bool comp = ATT && comp_on && (!SEL || !all_sel);
  float* csh = psm + lay.csh;  // [G][D]
  if (comp) {
    const int nk = p < nseg ? (nseg - 1 - p) / C + 1 : 0;
#pragma unroll 1
    for (int i4 = tid; i4 < G * D / 4; i4 += kPT) {
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
  if (tid == 0 && nown > 0 && (want_keys || ATT)) {
    if (!mbar_wait_bounded(bars + kPW, 0u, a.status, s, h, 20)) misc[kMBad] = 1;
  }
  __syncthreads();  // lse, zsl, ssl in place
  mark(0);

  // ---- a, b. keys, histograms, threshold
  int nsel_own = 0;
  uint32_t T = 0xFFFFFFFFu;
  int need = 0;
  bool take_all = true;
  const int need0 = K - 3;
  if (want_keys) {
    if (!all_sel) {
      for (int i = tid; i < kFine + 256; i += kPT) hf[i] = 0u;  // hf and he
      __syncthreads();
    }
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      const float lnn = ln_count(b == N - 1 ? L - kBlock * b : kBlock);
      float S = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float z = zsl[i * Gp + g], s2 = ssl[i * Gp + g];
        const float av = lnn + z + ((a.variant & kVarFirstOrderMass) ? 0.f : 0.5f * s2);
        const float ph = __expf(av - lse[g]);
        S = fmaf(ph, (a.variant & kVarNoVarianceFactor) ? 1.f : s2, S);
      }
      S = fmaxf(S, 0.f);
      const uint32_t key = __float_as_uint(S);
      keys[i] = key;
      if (a.scores) a.scores[(int64_t)u * a.score_stride + b] = S;
      if (!all_sel && b >= 1 && b <= N - 3) {
        atomicAdd(&hf[key >> kDigitShift], 1u);
        atomicAdd(&he[key >> 23], 1u);
      }
    }
    __syncthreads();
  }
  mark(1);
  cluster_wait();  // every peer's exchange histograms are zero
  if (SEL && !all_sel && need0 > 0) {
    // push this CTA's counts: the 16 fine bins of exponent e to rank e % C (no single rank
    // collects them all)
    {
      const int e = tid;  // kPT == 256 exponents
      if (he[e]) {
        const uint32_t fo = peer_smem(xfine + (e / C) * 16, (uint32_t)(e % C));
        const uint4* hv = reinterpret_cast<const uint4*>(hf + e * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = hv[k];
          if (v.x) red_peer_add(fo + 16u * k, v.x);
          if (v.y) red_peer_add(fo + 16u * k + 4u, v.y);
          if (v.z) red_peer_add(fo + 16u * k + 8u, v.z);
          if (v.w) red_peer_add(fo + 16u * k + 12u, v.w);
        }
      }
    }
    cluster_sync_all();  // barrier 1: rank e % C holds the cluster's 16 fine bins of exponent e
    mark(2);
    // thread t takes exponent 255 - t: its 16 fine bins from their owner, their sum scanned from
    // the top; the thread where the count of larger keys reaches K - 3 finds the fine bin
    const int ex = 255 - tid;
    uint32_t c16[16];
    {
      const uint32_t fo = peer_smem(xfine + (ex / C) * 16, (uint32_t)(ex % C));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = ld_peer_u4(fo + 16u * k);
        c16[4 * k] = v.x; c16[4 * k + 1] = v.y; c16[4 * k + 2] = v.z; c16[4 * k + 3] = v.w;
      }
    }
    int c = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) c += (int)c16[k];
    int tot;
    const int before = cta_exclusive_scan(c, misc + kMScan, &tot, lane, warp);
    if (before < need0 && need0 <= before + c) {
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
    T = (uint32_t)misc[kMT];
    need = need0 - misc[kMAbove];
    take_all = misc[kMCntT] == need;
  }
  mark(3);

  // ---- c. classification, the exchange of counts and tie lists, the selection
  int tot_sel = 0;     // selected blocks of the unit
  int sum_own = 0;     // of them in the CTAs' own lists (the rest are tie winners)
  int nwin = 0;
  int own_base = 0;    // offset of this CTA's part of the ascending selection
  const int nwo = (nown + 31) / 32;
  int* cnt = misc + kMCnt;  // [C] x (own count, tie count)
  if (SEL) {
    for (int w = tid; w < nwo; w += kPT) bits[w] = 0u;
    __syncthreads();
    for (int i = tid; i < nown; i += kPT) {
      const int b = b_lo + i;
      bool sl = all_sel || b == 0 || b >= N - 2;
      if (!sl && need0 > 0) {
        const uint32_t bin = keys[i] >> kDigitShift;
        if (bin > T || (bin == T && take_all)) {
          sl = true;
        } else if (bin == T) {
          const int slot = atomicAdd(misc + kMNtie, 1);
          if (slot < kTieCap) win[slot] = i;  // local indices of this CTA's tie candidates (win is free until the ranking)
        }
      }
      if (sl) atomicOr(&bits[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    if (warp == 0) {
      const int n = bitmap_list(bits, nwo, b_lo, own, nown < K ? nown : K, lane);
      if (lane == 0) misc[kMOwn] = n;
    }
    __syncthreads();
    nsel_own = misc[kMOwn];
    const int ntie = misc[kMNtie];
    if (!all_sel) {
      // push (own count, tie count) and the tie entries (key, block) to every CTA of the cluster
      if (tid < C) st_peer_u2(peer_smem(cnt + 2 * p, (uint32_t)tid), make_uint2((uint32_t)nsel_own, (uint32_t)ntie));
      const int nt = ntie < kTieCap ? ntie : kTieCap;
      for (int e = tid; e < nt * C; e += kPT) {
        const int q = e / nt, k = e % nt;
        const int i = win[k];
        st_peer_u2(peer_smem(tie + p * kTieCap + k, (uint32_t)q), make_uint2(keys[i], (uint32_t)(b_lo + i)));
      }
      if (ATT)
        for (int e = tid; e < nsel_own; e += kPT) {
          const int64_t row = row0 + own[e];
          prefetch_l2(a.k + row * kBlock * D, kBlock * D * 2);
          prefetch_l2(a.v + row * kBlock * D, kBlock * D * 2);
        }
      mark(4);
      cluster_sync_all();  // barrier 2: every CTA holds every count and tie list
      mark(5);
      // warp 0: prefix sums of the CTAs' counts (own lists, ties), their totals and the largest tie count
      int* opre = misc + kMOpre;
      int* tpre = misc + kMTpre;
      if (warp == 0) {
        const int co = lane < C ? cnt[2 * lane] : 0, ct = lane < C ? cnt[2 * lane + 1] : 0;
        int io = co, it = ct, mxl = ct;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, io, o), y2 = __shfl_up_sync(0xffffffffu, it, o);
          if (lane >= o) {
            io += y;
            it += y2;
          }
          mxl = max(mxl, __shfl_xor_sync(0xffffffffu, mxl, o));
        }
        if (lane <= C) {
          opre[lane] = io - co;
          tpre[lane] = it - ct;
        }
        if (lane == 31) {
          misc[kMSumOwn] = io;
          misc[kMNtAll] = it;
        }
        if (lane == 0) misc[kMMx] = mxl;
      }
      __syncthreads();
      sum_own = misc[kMSumOwn];
      const int nt_all = misc[kMNtAll], mx = misc[kMMx];
      if (!take_all && need > 0 && (mx > kTieCap || nt_all > kRankMax)) {
        // rare: resolve the threshold bin by more radix digits, then exchange the final counts
        refine_select(keys, bits, nown, b_lo, N, T, need, xref, lh, misc, C, p);
        if (warp == 0) {
          const int n = bitmap_list(bits, nwo, b_lo, own, nown < K ? nown : K, lane);
          if (lane == 0) misc[kMOwn] = n;
        }
        __syncthreads();
        nsel_own = misc[kMOwn];
        if (tid < C) st_peer_u2(peer_smem(cnt + 2 * p, (uint32_t)tid), make_uint2((uint32_t)nsel_own, 0u));
        cluster_sync_all();
        if (warp == 0) {
          const int co = lane < C ? cnt[2 * lane] : 0;
          int io = co;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, io, o);
            if (lane >= o) io += y;
          }
          if (lane <= C) opre[lane] = io - co;
          if (lane == 31) misc[kMSumOwn] = io;
        }
        __syncthreads();
        sum_own = misc[kMSumOwn];
        nwin = 0;
      } else if (!take_all && need > 0) {
        // rank every tie entry among all (key desc, block asc), one warp per entry over a
        // dense copy of the lists; the first `need` win, kept in rank order
        uint2* dense = reinterpret_cast<uint2*>(hf + 2 * kMaxC * kTieCap);
        for (int e = tid; e < C * kTieCap; e += kPT) {
          const int q = e / kTieCap, k = e % kTieCap;
          if (k < cnt[2 * q + 1]) dense[tpre[q] + k] = tie[e];
        }
        __syncthreads();
        for (int j = warp; j < nt_all; j += kPW) {
          const uint2 me = dense[j];
          int rank = 0;
          for (int j2 = lane; j2 < nt_all; j2 += 32) {
            const uint2 o = dense[j2];
            rank += (o.x > me.x) || (o.x == me.x && o.y < me.y);
          }
          rank = __reduce_add_sync(0xffffffffu, rank);
          if (lane == 0 && rank < need) win[rank] = (int)me.y;
        }
        nwin = need;
        __syncthreads();
      }
      tot_sel = sum_own + nwin;
      // this CTA's offset in the ascending selection: the lists of the lower ranks and the
      // tie winners below this CTA's blocks
      if (warp == 0) {
        int below = 0;
        for (int k = lane; k < nwin; k += 32) below += win[k] < b_lo;
        below = __reduce_add_sync(0xffffffffu, below);
        if (lane == 0) misc[kMWBelow] = below;
      }
      __syncthreads();
      own_base = opre[p] + misc[kMWBelow];
    } else {
      tot_sel = N;
      sum_own = N;
      own_base = b_lo;
    }
    // the ascending selection: this CTA's blocks and its tie winners, merged
    int* selrow = a.sel + (int64_t)u * K;
    for (int e = tid; e < nsel_own; e += kPT) {
      const int b = own[e];
      int pos = own_base + e;
      for (int k = 0; k < nwin; ++k) pos += (win[k] >= b_lo && win[k] < b);
      if (pos < K) selrow[pos] = b;
    }
    for (int k = tid; k < nwin; k += kPT) {
      const int b = win[k];
      if (b < b_lo || b >= b_hi) continue;
      int lo = 0, hi = nsel_own;  // own blocks below b (the list is ascending)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (own[mid] < b) lo = mid + 1; else hi = mid;
      }
      int pos = own_base + lo;
      for (int k2 = 0; k2 < nwin; ++k2) pos += (win[k2] >= b_lo && win[k2] < b);
      if (pos < K) selrow[pos] = b;
    }
    if (p == 0) {
      for (int i = tot_sel + tid; i < K; i += kPT) selrow[i] = -1;
      if (tid == 0 && tot_sel != (N < K ? N : K)) set_error(a.status, kDevInternal, s, h, 50);
    }
  } else {
    // the caller's selection: entries that are not ascending or not inside [0, N) are skipped and reported
    const int* selrow = a.sel + (int64_t)u * K;
    int bad = 0, cntv = 0;
    for (int i = tid; i < K; i += kPT) {
      const int e = __ldcg(selrow + i);
      const int prev = i > 0 ? __ldcg(selrow + i - 1) : -1;
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
  const unsigned long long t_sel = a.trace ? global_ns() : 0ull;
  if (tid == 0 && a.trace && a.P + (int)(gridDim.x + blockIdx.x) < a.trace_cap) {
    unsigned long long* rr = a.trace + 1 + 8 * (int64_t)(a.P + gridDim.x + blockIdx.x);
    rr[0] = ((unsigned long long)blockIdx.x << 32) | (2ull << 24) | (unsigned)misc[kMNtie];
#pragma unroll
    for (int k = 0; k < 7; ++k) rr[1 + k] = pmk[k];
  }
  if (SEL && !ATT) {
    // score/select only: no peer reads this CTA's shared memory after the barrier
    cluster_sync_all();
    if (tid == 0 && a.trace && a.P + (int)blockIdx.x < a.trace_cap) {
      unsigned long long* rr = a.trace + 1 + 8 * (int64_t)(a.P + blockIdx.x);
      rr[0] = ((unsigned long long)blockIdx.x << 32) | (1ull << 24) | (unsigned)p;
      rr[1] = (unsigned long long)u; rr[2] = t_start; rr[3] = t_wait; rr[4] = t_sel; rr[5] = t_sel;
    }
    return;
  }

  // ---- d. attention over this CTA's picks: positions (round * C + p) * kPW + warp of the selection
  // (the CTAs' own lists in rank order, then the tie winners; or the caller's list)
  const bool comp_blk = comp && tot_sel < N;
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
  const int hg = lane % G;  // head of this lane's softmax entries (lane, lane + 32, ...)
  uint32_t* wk = reinterpret_cast<uint32_t*>(psm + lay.stg + warp * lay.stg_w);
  uint32_t* wv = wk + kBlock * D / 2;
  float* wz = reinterpret_cast<float*>(wv + kBlock * D / 2);
  float* wp = wz + kBlock * G;
  uint32_t ph = 0u;
  const int slots_all = (SEL ? tot_sel : K);
  __syncthreads();  // the union switches from the selection to the attention staging
  for (int rnd = 0;; ++rnd) {
    const int j = (rnd * C + p) * kPW + warp;
    if (j >= slots_all || misc[kMBad] & 1) break;
    int b = -1;
    if (SEL) {
      if (all_sel) {
        b = j;
      } else if (j < sum_own) {
        const int* opre = misc + kMOpre;
        const unsigned bal = __ballot_sync(0xffffffffu, lane < C && opre[lane] <= j);
        const int q = 31 - __clz(bal);  // the highest CTA whose list starts at or before j
        b = (int)ld_peer_u32(peer_smem(own + (j - opre[q]), (uint32_t)q));
      } else {
        b = win[j - sum_own];
      }
    } else {
      const int* selrow = a.sel + (int64_t)u * K;
      const int e = __ldcg(selrow + j);
      const int prev = j > 0 ? __ldcg(selrow + j - 1) : -1;
      if (e >= 0 && e < N && (j == 0 || (prev >= 0 && prev < e))) b = e;
    }
    if (b < 0) continue;  // warp-uniform
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    const int64_t row = row0 + b;
    __syncwarp();  // the staging's previous contents are read
    if (lane == 0) {
      mbar_arrive_expect_tx(bars + warp, 2u * kBlock * D * 2u);
      const uint64_t pol = policy_evict_first();
      bulk_g2s_hint(wk, a.k + row * kBlock * D, kBlock * D * 2u, bars + warp, pol);
      bulk_g2s_hint(wv, a.v + row * kBlock * D, kBlock * D * 2u, bars + warp, pol);
    }
    float vbr[V];
#pragma unroll
    for (int i = 0; i < V; ++i) vbr[i] = comp_blk ? __ldcg(a.vbar + row * D + lane * V + i) : 0.f;
    // zbar of the block per head, as the stream left it
    const float zb_lane = (comp_blk && lane < G) ? __ldcg(a.zs + row * Gp + lane) : 0.f;
    if (!mbar_wait_bounded(bars + warp, ph, a.status, s, h, 62)) {
      mbar_drain_bounded(bars + warp);
      misc[kMBad] |= 1;
      break;
    }
    ph ^= 1u;
    // z = q . k / sqrt(d) of the block's tokens, TG tokens at a time
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
      // transposed reduction: lane j ends with the total of value j & (P - 1)
#pragma unroll
      for (int c = P; c > 1; c >>= 1) {
        const int off = c / 2;
        const bool up = (idx & off) != 0;
#pragma unroll
        for (int i = 0; i < c / 2; ++i) {
          const float send = up ? part[i] : part[i + c / 2];
          const float keep = up ? part[i + c / 2] : part[i];
          part[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
#pragma unroll
      for (int off = P; off < 32; off <<= 1) part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
      if (lane < P) wz[(gi * TG + jj) * G + gl] = part[0];
    }
    __syncwarp();
    // per head: the block's max, the running max and the rescale, p = e^(z - max) and its sum
    constexpr int EPL = (kBlock * G + 31) / 32;
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
    if (comp_blk) {
      // remove this block's own compensation term (the stream added it for every block)
      const float lnn = ln_count(n);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float e = lnn + __shfl_sync(0xffffffffu, zb_lane, g);
        const float mn = fmaxf(m[g], e);
        const float fo = (m[g] == -INFINITY) ? 0.f : __expf(m[g] - mn);
        const float fn = __expf(e - mn);
        m[g] = mn;
        l[g] = l[g] * fo - fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo - fn * vbr[i];
      }
    }
  }
  const unsigned long long t_att = a.trace ? global_ns() : 0ull;
  // ---- the CTA's partial: its warps and (warp 0's registers) its compensation share
  __syncthreads();  // the staging is free: the partials reuse the union
  float* red_a = psm + lay.red;            // [kPW][G][D]
  float* red_m = red_a + kPW * G * D;      // [kPW][G]
  float* red_l = red_m + kPW * G;          // [kPW][G]
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
  // per head, once: the common maximum of the warps' parts (and the compensation share)
  // and each part's factor (warp g: lane w takes warp w, lane kPW the share)
  float* fac = red_l + kPW * G;  // [G][kPW + 1] factors, then [G] maxima and [G] sums
  float* facM = fac + G * (kPW + 1);
  float* facL = facM + G;
  if (warp < G) {
    const int g = warp;
    const bool sh = lane == kPW && comp_blk;
    const float mw = lane < kPW ? red_m[lane * G + g] : (sh ? cR[g] : -INFINITY);
    const float lw = lane < kPW ? red_l[lane * G + g] : (sh ? cW[g] : 0.f);
    const float M = warp_max(mw);
    const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : __expf(mw - M);
    const float ls = warp_sum(lw * f);
    if (lane <= kPW) fac[g * (kPW + 1) + lane] = f;
    if (lane == 0) {
      facM[g] = M;
      facL[g] = ls;
    }
  }
  __syncthreads();
  // per float4 column item: combine, then push to the rank that merges it
  const int items = G * D / 4;
  const int ipr = post_ipr(D, G, C);
  for (int i4 = tid; i4 < items; i4 += kPT) {
    const int g = (4 * i4) / D, col = (4 * i4) % D;
    float4 as = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kPW; ++w) {
      const float f = fac[g * (kPW + 1) + w];
      const float4 x = *reinterpret_cast<const float4*>(red_a + (w * G + g) * D + col);
      as.x = fmaf(x.x, f, as.x);
      as.y = fmaf(x.y, f, as.y);
      as.z = fmaf(x.z, f, as.z);
      as.w = fmaf(x.w, f, as.w);
    }
    if (comp_blk) {
      const float f = fac[g * (kPW + 1) + kPW];
      const float4 x = *reinterpret_cast<const float4*>(csh + g * D + col);
      as.x = fmaf(x.x, f, as.x);
      as.y = fmaf(x.y, f, as.y);
      as.z = fmaf(x.z, f, as.z);
      as.w = fmaf(x.w, f, as.w);
    }
    const int rk = i4 / ipr, il = i4 - rk * ipr;
    const uint32_t dst = peer_smem(xm + (il * C + p) * 8, (uint32_t)rk);
    st_peer_f4(dst, as);
    st_peer_u2(dst + 16u, make_uint2(__float_as_uint(facM[g]), __float_as_uint(facL[g])));
  }
  cluster_sync_all();  // barrier 3: every partial of this rank's columns is here; no CTA touches a peer after this
  if (APPEND && p == 0 && tid == 0) {
    // every CTA of this cluster has read seq_len; the last cluster to get here
    // writes the lengths after this call's append (a sequence at capacity keeps its own)
    __threadfence();
    if (atomicAdd(a.arrive, 1) == (int)(gridDim.x / C) - 1) {
      for (int x = 0; x < a.B; ++x) {
        const bool f = ((x < 32 ? misc[kMFits] >> x : misc[kMFits + 1] >> (x - 32)) & 1) != 0;
        if (f) a.seq_len[x] = sL[x];
      }
      a.arrive[0] = 0;
      __threadfence();
    }
  }
  // this rank's column items: Cp (C rounded up to a power of two) lanes per item, lane q
  // takes CTA q's partial; the partials are merged across those lanes
  {
    const int i_lo = p * ipr, i_hi = min(items, i_lo + ipr);
    int Cp = 1;
    while (Cp < C) Cp <<= 1;
    const int nx = max(0, i_hi - i_lo) * Cp;  // groups of Cp lanes never straddle a warp (Cp divides 32)
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
      for (int o = 1; o < Cp; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = (M == -INFINITY || mq == -INFINITY) ? 0.f : __expf(mq - M);
      as.x *= f;
      as.y *= f;
      as.z *= f;
      as.w *= f;
      lq *= f;
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
  if (tid == 0 && a.trace && a.P + (int)blockIdx.x < a.trace_cap) {
    unsigned long long* rr = a.trace + 1 + 8 * (int64_t)(a.P + blockIdx.x);
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

template <int D, int G, int MODE>
static cudaError_t launch_post_mode(const LayerArgs& a, cudaStream_t st) {
  const void* fn = reinterpret_cast<const void*>(&k_post<D, G, MODE>);
  const size_t smem = (size_t)post_layout(D, G, a.C, a.bpc_max, a.K).total * 4;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (a.C > 8 && (e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess) return e;
  LayerArgs args = a;
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

}  // namespace compkv
