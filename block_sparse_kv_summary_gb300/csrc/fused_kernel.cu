// The CompKV decode step as one persistent, warp-specialised kernel.
//
// CompKV (onedev.kr/papers/157), section "무엇과 다른가": per (sequence, KV
// head) "unit", score every 16-token block from its summary, select the sink
// block, the two most recent blocks and the Top-K of S_b, then attend exactly
// to the selected blocks and add Mean compensation for the others under one
// normaliser.  Section "어떻게 쓰나" fuses the summary update of the open
// block with the K/V pack; here it is fused into the same launch as well.
//
// Work is a queue of tickets (one global atomic counter), written once at
// context creation in unit-major order:
//   S(u, c)  scoring item: blocks [64c, 64c + 64) of unit u;
//   A(u, p)  attention item: selected blocks [12p, 12p + 12) of unit u,
//            placed in the queue after the scoring items of unit u + 1.
// Each CTA = 1 producer warp + 12 consumer warps.  The producer claims
// tickets and stages a scoring item's kbar / vbar / Dbar rows into one of two
// shared-memory regions with 1-D bulk copies (cp.async.bulk, completion on an
// mbarrier), running up to two items ahead of the consumers.
//
// Scoring item (consumers): pass 1 zbar and sigma2 (a few lanes per block,
// shuffle-reduced), pass 2 per query head the item's logsumexp part of
// a = ln|b| + zbar + sigma2/2 and of the compensation weight ln|b| + zbar,
// pass 3 the item's compensation numerator sum_b |b| e^{zbar} vbar_b.  The
// item holding the newest token first appends it (new K/V written to the
// cache, the open block's summary recomputed from its tokens).  The CTA that
// completes the last scoring item of a unit (arrival counter) selects its
// blocks: LSE_g, S_b = sum_g phat sigma2, forced set, radix select with
// lower-index ties; then it publishes the unit as ready (epoch tag).
//
// Attention item: waits (bounded) for its unit, gathers its selected blocks'
// bf16 K/V (one block per warp), computes the exact softmax terms, removes
// each selected block's own Mean term (the scoring pass added one for every
// block), folds in its share of the per-item compensation sums, and writes a
// partial (m, l, acc); the last attention item of the unit merges them into
// out = acc / l.  If every block is selected, compensation is skipped.
//
// No wait depends on a ticket claimed later than the waiter's own, so the
// queue cannot deadlock whether or not all CTAs are resident; every wait is
// bounded and reports COMPKV_ERR_TIMEOUT through the status word.
#include "block_summary.cuh"
#include "compkv_launch.h"

namespace compkv {

constexpr int kCW = kAttendBlocks;       // consumer warps (one selected block each in an attention item)
constexpr int kCT = kCW * 32;            // consumer threads
constexpr int kFusedThreads = kCT + 32;  // + the producer warp
constexpr int kStages = 2;
constexpr int kBins = 2048;
constexpr int kListCap = 512;
constexpr int kItemScore = 0, kItemEnd = 2;  // attention items carry type 1
constexpr uint32_t kSpinLimit = 1u << 22;  // ~ a few hundred ms with the back-off below

struct Slot {
  int type, unit, index, L, N, b0, nb, append;
};

// ------------------------------------------------------------------ layout
__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline int fused_item_bytes(int D, int r) { return kChunk * (2 * D + r) * 4; }
__host__ __device__ inline int fused_select_bytes(int max_cap_blocks, int G) {
  const int nch = (max_cap_blocks + kChunk - 1) / kChunk;
  return align_up(max_cap_blocks, 4) * 4 + kBins * 4 + kListCap * 8 + align_up(nch * G, 4) * 4;
}
__host__ __device__ inline int fused_merge_bytes(int D, int G) { return kCW * G * (D + 2) * 4; }

struct FusedSmem {
  int region0, region1, q, qsq, zs, ss, ws, misc, bars, slots, total;
};

__host__ __device__ inline FusedSmem fused_layout(int D, int r, int G, int region_bytes) {
  FusedSmem L;
  int off = 0;
  L.region0 = off;
  off += region_bytes;
  L.region1 = off;
  off += region_bytes;
  L.q = off;
  off += G * D * 4;
  L.qsq = off;
  off += align_up(G * r, 4) * 4;
  L.zs = off;
  off += G * kChunk * 4;
  L.ss = off;
  off += G * kChunk * 4;
  L.ws = off;
  off += G * kChunk * 4;
  L.misc = off;
  off += 64 * 4;
  L.bars = align_up(off, 16);
  off = L.bars + 2 * kStages * 8;
  L.slots = align_up(off, 16);
  off = L.slots + kStages * (int)sizeof(Slot);
  L.total = align_up(off, 128);
  return L;
}

int fused_region_bytes(int D, int r, int G, int max_cap_blocks) {
  int R = fused_item_bytes(D, r);
  R = R > fused_select_bytes(max_cap_blocks, G) ? R : fused_select_bytes(max_cap_blocks, G);
  R = R > fused_merge_bytes(D, G) ? R : fused_merge_bytes(D, G);
  return align_up(R, 128);
}

size_t fused_smem_bytes(int D, int r, int G, int max_cap_blocks) {
  return (size_t)fused_layout(D, r, G, fused_region_bytes(D, r, G, max_cap_blocks)).total;
}

// misc ints in shared memory
enum Misc { kMFlag = 0, kMCount = 1, kMDigit = 2, kMAbove = 3, kMList = 4, kMBad = 5, kMScan = 8 /* 17 ints */,
            kMLse = 32 /* 8 floats */ };

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Exclusive prefix sum over the 512 consumer threads (one value each).
__device__ __forceinline__ int consumer_scan(int x, int* buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) buf[warp] = incl;
  consumer_sync();
  if (warp == 0) {
    const int v = lane < kCW ? buf[lane] : 0;
    int vi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) vi += y;
    }
    if (lane < kCW) buf[lane] = vi - v;
    if (lane == 31) buf[kCW] = vi;
  }
  consumer_sync();
  const int res = buf[warp] + incl - x;
  *total = buf[kCW];
  consumer_sync();
  return res;
}

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

// ================================================================== producer
template <int D, int G, int MODE>
__device__ void producer(const LayerArgs& a, unsigned char* sm, const FusedSmem& lay, uint64_t* full, uint64_t* empty,
                         Slot* slots) {
  constexpr bool COMP = (MODE & kFComp) != 0;
  constexpr bool SCORE = (MODE & kFScore) != 0;
  const int lane = threadIdx.x & 31;
  int st = 0;
  uint32_t uses[kStages] = {0, 0};
  for (;;) {
    int t = 0;
    if (lane == 0) t = atomicAdd(a.ticket, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    Slot sl{kItemEnd, 0, 0, 0, 0, 0, 0, 0};
    if (t < a.total_items) {
      const int code = __ldg(a.items + t);
      sl.type = (code >> 31) & 1;
      sl.unit = (code >> 20) & 0x7ff;
      sl.index = code & 0xfffff;
      const int s = sl.unit / a.Hkv;
      bool fits;
      sl.L = unit_tokens(a, s, (MODE & kFAppend) != 0, &fits);
      sl.N = ceil_blocks(sl.L);
      if (sl.type == kItemScore) {
        sl.b0 = sl.index * kChunk;
        sl.nb = sl.b0 < sl.N ? min(kChunk, sl.N - sl.b0) : 0;
        sl.append = ((MODE & kFAppend) && fits && sl.nb > 0 && sl.b0 + sl.nb == sl.N) ? 1 : 0;
      }
    }
    if (lane == 0) {
      mbar_wait_bounded(&empty[st], (uses[st] & 1) ^ 1, a.status, sl.unit, -1, 40);
      slots[st] = sl;
      uint32_t bytes = 0;
      const int nt = (sl.type == kItemScore) ? sl.nb - sl.append : 0;
      const bool dbar_bulk = SCORE && ((a.r & 3) == 0);
      if (nt > 0) {
        bytes = (uint32_t)nt * D * 4u * (COMP ? 2u : 1u);
        if (dbar_bulk) bytes += (uint32_t)nt * a.r * 4u;
      }
      mbar_arrive_expect_tx(&full[st], bytes);
      if (nt > 0) {
        const int s = sl.unit / a.Hkv, h = sl.unit % a.Hkv;
        const int64_t row0 = row_of(a, s, h, sl.b0);
        unsigned char* region = sm + (st == 0 ? lay.region0 : lay.region1);
        float* sk = reinterpret_cast<float*>(region);
        bulk_g2s(sk, a.kbar + row0 * D, (uint32_t)nt * D * 4u, &full[st]);
        if (COMP) bulk_g2s(sk + kChunk * D, a.vbar + row0 * D, (uint32_t)nt * D * 4u, &full[st]);
        if (dbar_bulk) bulk_g2s(sk + 2 * kChunk * D, a.dbar + row0 * a.r, (uint32_t)nt * a.r * 4u, &full[st]);
      }
    }
    __syncwarp();
    uses[st]++;
    st ^= 1;
    if (sl.type == kItemEnd) break;
  }
}

// ================================================================== selection (one unit)
template <int G>
__device__ void select_unit(const LayerArgs& a, int s, int h, int L, int N, unsigned char* region, int* misc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = chunk_record(a, s, h, 0);
  const int rs = rec_stride(a);
  uint32_t* keys = reinterpret_cast<uint32_t*>(region);
  uint32_t* hist = keys + align_up(a.cap_blocks[s], 4);
  uint32_t* lkey = hist + kBins;
  int* lidx = reinterpret_cast<int*>(lkey + kListCap);
  float* fch = reinterpret_cast<float*>(lidx + kListCap);
  float* lse = reinterpret_cast<float*>(misc + kMLse);
  int* selrow = a.sel + ((int64_t)s * a.Hkv + h) * K;

  // 1. LSE_g from the items' (max, sum) pairs
  if (warp < G) {
    const int g = warp;
    float M = -INFINITY, S = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const float* rg = a.chunk_rec + (int64_t)(rec0 + c) * rs + g * (4 + a.d);
      const float mc = __ldcg(rg), lc = __ldcg(rg + 1);
      if (mc > M) {
        S = S * expf(M - mc) + lc;
        M = mc;
      } else {
        S += lc * expf(mc - M);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o), S2 = __shfl_xor_sync(0xffffffffu, S, o);
      const float Mn = fmaxf(M, M2);
      S = (M == -INFINITY ? 0.f : S * expf(M - Mn)) + (M2 == -INFINITY ? 0.f : S2 * expf(M2 - Mn));
      M = Mn;
    }
    if (lane == 0) lse[g] = M + logf(S);
  }
  consumer_sync();
  // 2. per-item factors exp(m_a - LSE_g)
  for (int i = tid; i < nch * G; i += kCT) {
    const int c = i / G, g = i % G;
    fch[i] = expf(__ldcg(a.chunk_rec + (int64_t)(rec0 + c) * rs + g * (4 + a.d)) - lse[g]);
  }
  for (int i = tid; i < kBins; i += kCT) hist[i] = 0;
  consumer_sync();
  // 3. S_b as order-preserving uint32 keys
  float* scores = a.scores ? a.scores + ((int64_t)s * a.Hkv + h) * a.score_stride : nullptr;
  for (int b = tid; b < N; b += kCT) {
    const int c = b / kChunk, o = b % kChunk;
    float S = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) S = fmaf(__ldcg(a.chunk_u + ((int64_t)(rec0 + c) * G + g) * kChunk + o), fch[c * G + g], S);
    S = fmaxf(S, 0.f);
    keys[b] = __float_as_uint(S);
    if (scores) scores[b] = S;
  }
  consumer_sync();
  if (N <= K) {
    for (int i = tid; i < K; i += kCT) selrow[i] = i < N ? i : -1;
    return;
  }
  // 4. radix select of the K-3 largest candidates (blocks 1..N-3), 11/11/10-bit digits
  int need = K - 3;
  uint32_t prefix = 0, pmask = 0;
  bool done = need == 0;
  const int cand_lo = 1, cand_hi = N - 3;  // inclusive
  for (int level = 0; level < 3 && !done; ++level) {
    const int shift = level == 0 ? 21 : (level == 1 ? 10 : 0);
    const int nbins = level == 2 ? 1024 : 2048;
    const uint32_t dmask = (uint32_t)nbins - 1;
    if (level > 0) {
      for (int i = tid; i < kBins; i += kCT) hist[i] = 0;
      consumer_sync();
    }
    for (int b = cand_lo + tid; b <= cand_hi; b += kCT) {
      const uint32_t key = keys[b];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
    }
    consumer_sync();
    {
      // thread t owns `per` consecutive bins of the descending order
      const int per = (nbins + kCT - 1) / kCT;
      int loc = 0;
      for (int i = 0; i < per; ++i) {
        const int bin = nbins - 1 - per * tid - i;
        if (bin >= 0) loc += (int)hist[bin];
      }
      int total;
      const int before = consumer_scan(loc, misc + kMScan, &total);
      if (before < need && need <= before + loc) {
        int run = before;
        for (int i = 0; i < per; ++i) {
          const int bin = nbins - 1 - per * tid - i;
          if (bin < 0) break;
          const int c = (int)hist[bin];
          if (run < need && need <= run + c) {
            misc[kMDigit] = bin;
            misc[kMAbove] = run;
          }
          run += c;
        }
      }
      if (tid == 0) misc[kMList] = 0;
    }
    consumer_sync();
    const uint32_t Dg = (uint32_t)misc[kMDigit];
    const int above = misc[kMAbove];
    const int cntD = (int)hist[Dg];
    // every candidate above the threshold digit is selected
    for (int b = cand_lo + tid; b <= cand_hi; b += kCT) {
      const uint32_t key = keys[b];
      if ((key & pmask) == prefix && ((key >> shift) & dmask) > Dg) keys[b] = key | 0x80000000u;
    }
    need -= above;
    prefix |= Dg << shift;
    pmask |= dmask << shift;
    if (cntD == need) {
      for (int b = cand_lo + tid; b <= cand_hi; b += kCT)
        if ((keys[b] & pmask) == prefix) keys[b] |= 0x80000000u;
      done = true;
    } else if (cntD <= kListCap) {
      for (int b = cand_lo + tid; b <= cand_hi; b += kCT) {
        const uint32_t key = keys[b];
        if ((key & pmask) == prefix) {
          const int p = atomicAdd(misc + kMList, 1);
          lkey[p] = key;
          lidx[p] = b;
        }
      }
      consumer_sync();
      const int n = misc[kMList];
      if (tid < n) {
        const uint32_t k0 = lkey[tid];
        const int i0 = lidx[tid];
        int rank = 0;
        for (int f = 0; f < n; ++f) {
          const uint32_t kf = lkey[f];
          rank += (kf > k0) || (kf == k0 && lidx[f] < i0);
        }
        if (rank < need) keys[i0] = k0 | 0x80000000u;
      }
      done = true;
    }
    consumer_sync();
  }
  if (!done) {
    // all remaining candidates carry the same key: take the `need` lowest indices
    const int span = cand_hi - cand_lo + 1;
    const int per = (span + kCT - 1) / kCT;
    const int lo = cand_lo + min(span, tid * per), hi = cand_lo + min(span, tid * per + per);
    int cnt = 0;
    for (int b = lo; b < hi; ++b) cnt += (keys[b] & pmask) == prefix;
    int total;
    int rk = consumer_scan(cnt, misc + kMScan, &total);
    for (int b = lo; b < hi; ++b)
      if ((keys[b] & pmask) == prefix) {
        if (rk < need) keys[b] |= 0x80000000u;
        ++rk;
      }
    consumer_sync();
  }
  if (tid == 0) {
    keys[0] |= 0x80000000u;
    keys[N - 2] |= 0x80000000u;
    keys[N - 1] |= 0x80000000u;
  }
  consumer_sync();
  // 5. ascending compaction
  {
    const int per = (N + kCT - 1) / kCT;
    const int lo = min(N, tid * per), hi = min(N, tid * per + per);
    int cnt = 0;
    for (int b = lo; b < hi; ++b) cnt += keys[b] >> 31;
    int total;
    int pos = consumer_scan(cnt, misc + kMScan, &total);
    if (tid == 0 && total != K) set_error(a.status, kDevInternal, s, h, 50);
    for (int b = lo; b < hi; ++b)
      if ((keys[b] >> 31) && pos < K) selrow[pos++] = b;
  }
}

// ================================================================== scoring item
template <int D, int G, int MODE>
__device__ void score_item(const LayerArgs& a, const Slot& sl, unsigned char* region, unsigned char* sm,
                           const FusedSmem& lay) {
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv;
  const int r = a.r;
  const int L = sl.L, N = sl.N, nb = sl.nb, b0 = sl.b0;
  const int rec = chunk_record(a, s, h, sl.index);
  int* misc = reinterpret_cast<int*>(sm + lay.misc);
  if (nb > 0) {
    float* sk = reinterpret_cast<float*>(region);
    float* sv = sk + kChunk * D;
    float* sd = sv + kChunk * D;
    float* sq = reinterpret_cast<float*>(sm + lay.q);
    float* sqsq = reinterpret_cast<float*>(sm + lay.qsq);
    float* zs = reinterpret_cast<float*>(sm + lay.zs);
    float* ss = reinterpret_cast<float*>(sm + lay.ss);
    float* ws = reinterpret_cast<float*>(sm + lay.ws);
    const int64_t row0 = row_of(a, s, h, b0);
    const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
    for (int i = tid; i < G * D; i += kCT) sq[i] = qg[i];
    if (SCORE && (r & 3))
      for (int i = tid; i < (nb - sl.append) * r; i += kCT) sd[i] = a.dbar[row0 * r + i];
    if (sl.append && warp == 0) {
      // pack the new token and recompute the open block's summary (into the
      // staged rows and back to the cache)
      constexpr int V = D / 32;
      const int b = N - 1, n = L - kBlock * b;
      const int64_t row = row0 + (nb - 1);
      const __nv_bfloat16* kn = a.k_new + ((int64_t)s * a.Hkv + h) * D;
      const __nv_bfloat16* vn = a.v_new + ((int64_t)s * a.Hkv + h) * D;
      store_bf16_raw<V>(a.k + (row * kBlock + n - 1) * D + lane * V, kn + lane * V);
      store_bf16_raw<V>(a.v + (row * kBlock + n - 1) * D + lane * V, vn + lane * V);
      float* kb = sk + (nb - 1) * D;
      float* vb = sv + (nb - 1) * D;
      float* db = sd + (nb - 1) * r;
      warp_block_summary<D>(a.k + row * kBlock * D, a.v + row * kBlock * D, n, kn, vn, kb, vb, db, r, lane);
      __syncwarp();
      for (int i = lane; i < D; i += 32) {
        a.kbar[row * D + i] = kb[i];
        a.vbar[row * D + i] = vb[i];
      }
      for (int i = lane; i < r; i += 32) a.dbar[row * r + i] = db[i];
    }
    consumer_sync();
    if (SCORE) {
      const int gs = D / r;
      for (int i = tid; i < G * r; i += kCT) {
        const int g = i / r, t = i % r;
        float acc = 0.f;
        for (int j = 0; j < gs; ++j) {
          const float x = sq[g * D + t * gs + j];
          acc = fmaf(x, x, acc);
        }
        sqsq[i] = acc;
      }
      consumer_sync();
    }
    // ---- pass 1: zbar (and sigma2) with LPB lanes per block
    {
      constexpr int LPB = (G * D / 16 > 32) ? 32 : 16;
      constexpr int NV = D / LPB;
      constexpr int BPW = 32 / LPB;
      const int j = lane % LPB, sub = lane / LPB;
      auto coord = [&](int i) -> int {
        if (NV == 8) return i < 4 ? 4 * j + i : D / 2 + 4 * j + (i - 4);
        return NV * j + i;
      };
      float qr[G][NV];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < NV; ++i) qr[g][i] = sq[g * D + coord(i)];
      for (int base = warp * BPW; base < nb; base += kCW * BPW) {
        const int blk = base + sub;
        const bool valid = blk < nb;
        const int rb = valid ? blk : base;
        float kv[NV];
        if (NV == 8) {
          const float4 x = *reinterpret_cast<const float4*>(sk + rb * D + 4 * j);
          const float4 y = *reinterpret_cast<const float4*>(sk + rb * D + D / 2 + 4 * j);
          kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w;
          kv[4 % NV] = y.x; kv[5 % NV] = y.y; kv[6 % NV] = y.z; kv[7 % NV] = y.w;
        } else if (NV == 4) {
          const float4 x = *reinterpret_cast<const float4*>(sk + rb * D + 4 * j);
          kv[0] = x.x; kv[1] = x.y; kv[2 % NV] = x.z; kv[3 % NV] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(sk + rb * D + 2 * j);
          kv[0] = x.x; kv[1 % NV] = x.y;
        }
        float zacc[G], sacc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          zacc[g] = 0.f;
          sacc[g] = 0.f;
#pragma unroll
          for (int i = 0; i < NV; ++i) zacc[g] = fmaf(qr[g][i], kv[i], zacc[g]);
        }
        if (SCORE) {
          for (int t = j; t < r; t += LPB) {
            const float dv = sd[rb * r + t];
#pragma unroll
            for (int g = 0; g < G; ++g) sacc[g] = fmaf(sqsq[g * r + t], dv, sacc[g]);
          }
        }
#pragma unroll
        for (int o = LPB / 2; o > 0; o >>= 1) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            zacc[g] += __shfl_xor_sync(0xffffffffu, zacc[g], o);
            if (SCORE) sacc[g] += __shfl_xor_sync(0xffffffffu, sacc[g], o);
          }
        }
        if (j == 0 && valid) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            zs[g * kChunk + blk] = zacc[g] * InvSqrt<D>::v;
            if (SCORE) ss[g * kChunk + blk] = sacc[g] / (float)D;
          }
        }
      }
    }
    consumer_sync();
    // ---- pass 2: one warp per query head
    if (warp < G) {
      const int g = warp;
      float av[2], cv[2];
      float ma = -INFINITY, mc = -INFINITY;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int blk = lane + 32 * i;
        av[i] = cv[i] = -INFINITY;
        if (blk < nb) {
          const int bb = b0 + blk;
          const int n = (bb == N - 1) ? L - kBlock * bb : kBlock;
          cv[i] = ln_n(n) + zs[g * kChunk + blk];
          if (SCORE) av[i] = cv[i] + 0.5f * ss[g * kChunk + blk];
        }
        ma = fmaxf(ma, av[i]);
        mc = fmaxf(mc, cv[i]);
      }
      float la = 0.f, lc = 0.f;
      if (SCORE) {
        ma = warp_max(ma);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
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
        for (int i = 0; i < 2; ++i) {
          const int blk = lane + 32 * i;
          const float w = (blk < nb) ? expf(cv[i] - mc) : 0.f;
          lc += w;
          ws[g * kChunk + blk] = w;
          a.chunk_z[((int64_t)rec * G + g) * kChunk + blk] = (blk < nb) ? zs[g * kChunk + blk] : 0.f;
        }
        lc = warp_sum(lc);
      }
      if (lane == 0) {
        float* rg = a.chunk_rec + (int64_t)rec * rec_stride(a) + g * (4 + D);
        rg[0] = ma;
        rg[1] = la;
        rg[2] = mc;
        rg[3] = lc;
      }
    }
    // ---- pass 3: compensation numerator sum_b w_{g,b} vbar_b
    if (COMP) {
      consumer_sync();
      constexpr int V = D / 32;
      float acc[G][V];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
      for (int blk = warp; blk < nb; blk += kCW) {
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
          const float w = ws[g * kChunk + blk];
#pragma unroll
          for (int i = 0; i < V; ++i) acc[g][i] = fmaf(w, vv[i], acc[g][i]);
        }
      }
      consumer_sync();
      float* red = sk;  // [kCW][G][D], reuses the staged rows
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < V; ++i) red[(warp * G + g) * D + lane * V + i] = acc[g][i];
      consumer_sync();
      float* rp = a.chunk_rec + (int64_t)rec * rec_stride(a);
      for (int i = tid; i < G * D; i += kCT) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kCW; ++w) t += red[w * G * D + i];
        rp[(i / D) * (4 + D) + 4 + (i % D)] = t;
      }
    }
  }
  // ---- arrival: the last scoring item of the unit selects and publishes it
  __threadfence();
  consumer_sync();
  if (tid == 0) {
    const int prev = atomicAdd(a.bcount + u, 1);
    const int last = prev == a.nchunk[s] - 1;
    if (last) a.bcount[u] = 0;
    misc[kMFlag] = last;
  }
  consumer_sync();
  if (misc[kMFlag]) {
    __threadfence();
    if (MODE & kFSelect) select_unit<G>(a, s, h, L, N, region, misc);
    __threadfence();
    consumer_sync();
    if (tid == 0) st_release(a.ready + u, a.epoch);
  }
}

// ================================================================== attention item
// Sum of 32 (or 16) values across the warp: lane l ends with the total of value
// index l % P.  31 shuffles.
template <int P>
__device__ __forceinline__ float transpose_reduce(float (&v)[P], int lane) {
  if (P == 16) {
#pragma unroll
    for (int i = 0; i < P; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 16);
  }
#pragma unroll
  for (int off = (P == 32 ? 16 : 8), c = P; off > 0; off >>= 1, c >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float send = upper ? v[i] : v[i + c / 2];
      const float keep = upper ? v[i + c / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

__device__ __forceinline__ void fold(float& m, float& l, float e, float& fo, float& fn) {
  const float mn = fmaxf(m, e);
  fo = (m == -INFINITY) ? 0.f : expf(m - mn);
  fn = expf(e - mn);
  m = mn;
}

template <int D, int G, int MODE>
__device__ void attend_item(const LayerArgs& a, const Slot& sl, unsigned char* region, unsigned char* sm,
                            const FusedSmem& lay) {
  constexpr int V = D / 32;
  constexpr int TG = (32 / G) > 16 ? 16 : (32 / G);  // tokens per reduction group
  constexpr int P = TG * G;                          // 16 or 32 values per group
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv, p = sl.index;
  const int L = sl.L, N = sl.N, K = a.K;
  int* misc = reinterpret_cast<int*>(sm + lay.misc);

  // wait until the unit is scored (and selected)
  if (tid == 0) {
    misc[kMFlag] = 0;
    misc[kMCount] = 0;
    misc[kMBad] = 0;
    uint32_t it = 0;
    while (ld_acquire(a.ready + u) != a.epoch) {
      if (++it > kSpinLimit) {
        set_error(a.status, kDevTimeout, s, h, 60);
        misc[kMFlag] = 1;
        break;
      }
      __nanosleep(64);
    }
  }
  consumer_sync();
  __threadfence();
  const bool timed_out = misc[kMFlag] != 0;
  const int* selrow = a.sel + ((int64_t)s * a.Hkv + h) * K;
  {
    int cnt = 0, bad = 0;
    for (int i = tid; i < K; i += kCT) {
      const int e = __ldcg(selrow + i);
      const int prev = i > 0 ? __ldcg(selrow + i - 1) : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      cnt += ok;
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cnt) atomicAdd(misc + kMCount, cnt);
      if (bad) misc[kMBad] = 1;
    }
  }
  consumer_sync();
  const int nsel = misc[kMCount];
  if (misc[kMBad] && p == 0 && tid == 0) set_error(a.status, kDevBadSelection, s, h, 61);
  const bool comp = nsel < N && !timed_out;

  float qr[G][V];
  const float* qg = a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) qr[g][i] = qg[g * D + lane * V + i] * InvSqrt<D>::v;
  float m[G], l[G], acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  }

  // this warp's selected block
  const int my_i = p * kCW + warp;
  int b = -1;
  if (!timed_out && my_i < K) {
    const int e = __ldcg(selrow + my_i);
    const int prev = my_i > 0 ? __ldcg(selrow + my_i - 1) : -1;
    if (e >= 0 && e < N && (my_i == 0 || (prev >= 0 && prev < e))) b = e;
  }
  if (b >= 0) {
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    const int64_t row = row_of(a, s, h, b);
    const __nv_bfloat16* kp = a.k + row * kBlock * D + lane * V;
    const __nv_bfloat16* vp = a.v + row * kBlock * D + lane * V;
    for (int j0 = 0; j0 < kBlock; j0 += TG) {
      float part[P];
#pragma unroll
      for (int jj = 0; jj < TG; ++jj) {
        float kf[V];
        if (V == 4) {
          const uint2 w = __ldcg(reinterpret_cast<const uint2*>(kp + (j0 + jj) * D));
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
          const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
          kf[0] = x.x; kf[1] = x.y; kf[2 % V] = y.x; kf[3 % V] = y.y;
        } else {
          const unsigned w = __ldcg(reinterpret_cast<const unsigned*>(kp + (j0 + jj) * D));
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
          kf[0] = x.x; kf[1 % V] = x.y;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float t = 0.f;
#pragma unroll
          for (int i = 0; i < V; ++i) t = fmaf(qr[g][i], kf[i], t);
          part[jj * G + g] = t;
        }
      }
      const float z = transpose_reduce<P>(part, lane);
      const int idx = lane & (P - 1);
      const int jj = idx / G, gl = idx % G;
      const bool valid = j0 + jj < n;
      // group max per query head
      float gm = valid ? z : -INFINITY;
#pragma unroll
      for (int o = G; o < P; o <<= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      float mn_l = 0.f;
      float scale[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float gmg = __shfl_sync(0xffffffffu, gm, g);
        const float mn = fmaxf(m[g], gmg);
        scale[g] = (m[g] == -INFINITY) ? 0.f : expf(m[g] - mn);
        m[g] = mn;
        if (g == gl) mn_l = mn;
      }
      const float pz = valid ? expf(z - mn_l) : 0.f;
      float ps = pz;
#pragma unroll
      for (int o = G; o < P; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        l[g] = l[g] * scale[g] + __shfl_sync(0xffffffffu, ps, g);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] *= scale[g];
      }
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        float vf[V];
        if (V == 4) {
          const uint2 w = __ldcg(reinterpret_cast<const uint2*>(vp + (j0 + t) * D));
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
          const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
          vf[0] = x.x; vf[1] = x.y; vf[2 % V] = y.x; vf[3 % V] = y.y;
        } else {
          const unsigned w = __ldcg(reinterpret_cast<const unsigned*>(vp + (j0 + t) * D));
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
          vf[0] = x.x; vf[1 % V] = x.y;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = __shfl_sync(0xffffffffu, pz, t * G + g);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[g][i] = fmaf(pg, vf[i], acc[g][i]);
        }
      }
    }
    if (comp) {
      // remove this block's own Mean compensation term
      const int c = b / kChunk, o = b % kChunk;
      const int rec = chunk_record(a, s, h, c);
      const float lnn = ln_n(n);
      float vb[V];
#pragma unroll
      for (int i = 0; i < V; ++i) vb[i] = __ldcg(a.vbar + row * D + lane * V + i);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float e = lnn + __ldcg(a.chunk_z + ((int64_t)rec * G + g) * kChunk + o);
        float fo, fn;
        fold(m[g], l[g], e, fo, fn);
        l[g] = l[g] * fo - fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo - fn * vb[i];
      }
    }
  }
  // this item's share of the scoring items' compensation sums
  if (comp) {
    const int nch = (N + kChunk - 1) / kChunk;
    const int c0 = (int)((int64_t)p * nch / a.splits), c1 = (int)((int64_t)(p + 1) * nch / a.splits);
    for (int c = c0 + warp; c < c1; c += kCW) {
      const float* rp = a.chunk_rec + (int64_t)chunk_record(a, s, h, c) * rec_stride(a);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float mc = __ldcg(rp + g * (4 + D) + 2);
        const float lc = __ldcg(rp + g * (4 + D) + 3);
        float fo, fn;
        fold(m[g], l[g], mc, fo, fn);
        l[g] = l[g] * fo + lc * fn;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = acc[g][i] * fo + __ldcg(rp + g * (4 + D) + 4 + lane * V + i) * fn;
      }
    }
  }
  // merge the warps: red_m[kCW][G], red_l[kCW][G], red_a[kCW][G][D]
  float* red_m = reinterpret_cast<float*>(region);
  float* red_l = red_m + kCW * G;
  float* red_a = red_l + kCW * G;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      red_m[warp * G + g] = m[g];
      red_l[warp * G + g] = l[g];
    }
#pragma unroll
    for (int i = 0; i < V; ++i) red_a[(warp * G + g) * D + lane * V + i] = acc[g][i];
  }
  consumer_sync();
  const int unit_rec = u * a.splits;
  float* srec = a.split_rec + (int64_t)(unit_rec + p) * rec_stride(a);
  for (int idx = tid; idx < G * D; idx += kCT) {
    const int g = idx / D, col = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCW; ++w) M = fmaxf(M, red_m[w * G + g]);
    float ls = 0.f, as = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCW; ++w) {
        const float mw = red_m[w * G + g];
        const float f = (mw == -INFINITY) ? 0.f : expf(mw - M);
        ls += red_l[w * G + g] * f;
        as += red_a[(w * G + g) * D + col] * f;
      }
    }
    if (col == 0) {
      srec[g * (4 + D)] = M;
      srec[g * (4 + D) + 1] = ls;
    }
    srec[g * (4 + D) + 4 + col] = as;
  }
  // the last attention item of the unit merges all of them
  __threadfence();
  consumer_sync();
  if (tid == 0) {
    const int prev = atomicAdd(a.dcount + u, 1);
    const int last = prev == a.splits - 1;
    if (last) a.dcount[u] = 0;
    misc[kMFlag] = last;
  }
  consumer_sync();
  if (!misc[kMFlag]) return;
  __threadfence();
  const float* recs = a.split_rec + (int64_t)unit_rec * rec_stride(a);
  float* out = a.out + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
  const int rs = rec_stride(a);
  for (int idx = tid; idx < G * D; idx += kCT) {
    const int g = idx / D, col = idx % D;
    float M = -INFINITY, ls = 0.f, as = 0.f;
    for (int q0 = 0; q0 < a.splits; q0 += 8) {
      float mv[8], lv[8], av[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int pp = q0 + k;
        if (pp < a.splits) {
          const float* rp = recs + (int64_t)pp * rs + g * (4 + D);
          mv[k] = __ldcg(rp);
          lv[k] = __ldcg(rp + 1);
          av[k] = __ldcg(rp + 4 + col);
        } else {
          mv[k] = -INFINITY;
          lv[k] = av[k] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (mv[k] == -INFINITY) continue;
        const float mn = fmaxf(M, mv[k]);
        const float fo = (M == -INFINITY) ? 0.f : expf(M - mn);
        const float fn = expf(mv[k] - mn);
        ls = ls * fo + lv[k] * fn;
        as = as * fo + av[k] * fn;
        M = mn;
      }
    }
    out[g * D + col] = (ls > 0.f) ? as / ls : 0.f;
  }
}

// ================================================================== kernel
template <int D, int G, int MODE>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_kernel(LayerArgs a) {
  extern __shared__ __align__(128) unsigned char sm[];
  const FusedSmem lay = fused_layout(D, a.r, G, a.region_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + lay.bars);
  uint64_t* empty = full + kStages;
  Slot* slots = reinterpret_cast<Slot*>(sm + lay.slots);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= kCT) {
    producer<D, G, MODE>(a, sm, lay, full, empty, slots);
  } else {
    int st = 0;
    uint32_t uses[kStages] = {0, 0};
    for (;;) {
      mbar_wait_bounded(&full[st], uses[st] & 1, a.status, -1, -1, 41);
      const Slot sl = slots[st];
      if (sl.type == kItemEnd) break;
      unsigned char* region = sm + (st == 0 ? lay.region0 : lay.region1);
      if (sl.type == kItemScore)
        score_item<D, G, MODE>(a, sl, region, sm, lay);
      else if (MODE & kFAttend)
        attend_item<D, G, MODE>(a, sl, region, sm, lay);
      consumer_sync();
      if (tid == 0) mbar_arrive(&empty[st]);
      uses[st]++;
      st ^= 1;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(a.done, 1);
    if (prev == (int)gridDim.x - 1) {
      // every CTA has left the queue: reset it and publish the new lengths
      *a.ticket = 0;
      *a.done = 0;
      if (MODE & kFAppend) {
        for (int s = 0; s < a.B; ++s) {
          const int Lold = a.seq_len[s];
          if (Lold >= 0 && Lold < a.cap_blocks[s] * kBlock)
            a.seq_len[s] = Lold + 1;
          else
            set_error(a.status, kDevCapacity, s, -1, 42);
        }
      }
      __threadfence();
    }
  }
}

template <int D, int G, int MODE>
static cudaError_t launch_fused_dgm(const LayerArgs& a, int grid, cudaStream_t st) {
  const size_t sm = (size_t)fused_layout(D, a.r, G, a.region_bytes).total;
  cudaError_t e = cudaFuncSetAttribute(fused_kernel<D, G, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  fused_kernel<D, G, MODE><<<grid, kFusedThreads, sm, st>>>(a);
  return cudaGetLastError();
}

template <int D, int G>
static cudaError_t launch_fused_dg(const LayerArgs& a, int mode, int grid, cudaStream_t st) {
  switch (mode) {
    case kFusedDecode: return launch_fused_dgm<D, G, kFusedDecode>(a, grid, st);
    case kFusedScoreSelect: return launch_fused_dgm<D, G, kFusedScoreSelect>(a, grid, st);
    case kFusedAttend: return launch_fused_dgm<D, G, kFusedAttend>(a, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fused(const LayerArgs& a, int mode, int grid, cudaStream_t st) {
#define COMPKV_G(DD)                                          \
  switch (a.G) {                                              \
    case 1: return launch_fused_dg<DD, 1>(a, mode, grid, st); \
    case 2: return launch_fused_dg<DD, 2>(a, mode, grid, st); \
    case 4: return launch_fused_dg<DD, 4>(a, mode, grid, st); \
    case 8: return launch_fused_dg<DD, 8>(a, mode, grid, st); \
    default: return cudaErrorInvalidValue;                    \
  }
  if (a.d == 128) {
    COMPKV_G(128)
  } else {
    COMPKV_G(64)
  }
#undef COMPKV_G
}

}  // namespace compkv
