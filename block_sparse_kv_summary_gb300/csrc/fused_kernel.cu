// The CompKV decode step as one persistent, warp-specialised kernel.
//
// CompKV (onedev.kr/papers/157), section "무엇과 다른가": per (sequence, KV
// head) "unit", score every 16-token block from its summary, select the sink
// block, the two most recent blocks and the Top-K of S_b, then attend exactly
// to the selected blocks and add Mean compensation for the others under one
// normaliser.  Section "어떻게 쓰나" fuses the summary update of the open
// block with the K/V pack; here it joins the same launch.
//
// Two phases.  The selection needs only kbar and Dbar; vbar is needed only
// for the compensation.  So the work queue (one global ticket counter,
// written once per context) lists
//   phase 1: S(u, c)  scoring: kbar, Dbar of blocks [64c, 64c + 64) of unit u,
//            for every unit (unit-major);
//   phase 2: A(u, p)  attention: selected blocks [12p, 12p + 12) of unit u,
//            C(u, c)  compensation: vbar of blocks [128c, 128c + 128),
// and a unit's selection runs while phase 2 of the earlier units streams:
// its latency hides behind the vbar reads instead of adding to the step.
//
// CTA = 1 producer thread (warp 12) + 12 consumer warps.  The producer claims
// tickets, stages S and C items' summary rows into a ring of 2-3 shared-memory
// regions with 1-D bulk copies (cp.async.bulk, completion on an mbarrier),
// and counts completed items per unit.  When a unit's last scoring item
// completes it queues a SELECT follow-up in its own ring; when its last
// attention / compensation item completes, a MERGE follow-up.  Before its
// first phase-2 item a producer settles the counts of everything it has
// published, so no phase-2 item (which waits for its unit's selection) can
// sit in a ring ahead of a SELECT that it waits for.  Every wait is bounded
// and reports COMPKV_ERR_TIMEOUT through the status word.
//
// Numerics (fp32 throughout, summaries and logits from the exact bf16 K/V):
//   S item:  zbar = q.kbar/sqrt(d); sigma2 = (1/d) sum_t Qsq_t Dbar_t;
//            a = ln|b| + zbar + sigma2/2; per item and query head the max of
//            a, sum e^(a - max), and u = e^(a - max) sigma2 per block.
//   SELECT:  LSE_g from the items' pairs; S_b = sum_g u exp(max_item - LSE_g)
//            = sum_g phat sigma2; radix Top-K on the bits of S_b (>= 0), ties
//            to the lower index; ascending list + bitmap; the compensation
//            reference M_g = max_b (ln|b| + zbar_{g,b}).
//   A item:  exact softmax terms of the selected blocks' tokens -> (m, l, acc).
//   C item:  w = e^(ln|b| + zbar - M_g) (<= 1) for unselected blocks,
//            sum_b w vbar_b and sum_b w added (fp32 atomics) to the unit's
//            accumulator.
//   MERGE:   out = (sum_p e^(m_p - R) acc_p + e^(M_g - R) sum w vbar)
//                / (sum_p e^(m_p - R) l_p   + e^(M_g - R) sum w).
// If every block is selected there is nothing to compensate.
#include "block_summary.cuh"
#include "compkv_launch.h"

namespace compkv {

constexpr int kCW = kAttendBlocks;       // consumer warps (one selected block each in an attention item)
constexpr int kCT = kCW * 32;            // consumer threads
constexpr int kFusedThreads = kCT + 32;  // + the producer warp
constexpr int kMaxStages = 3;
constexpr int kBins = 4096;     // shared histogram of the radix select
constexpr int kPrivBins = 256;  // per-warp histogram of its first (exponent) digit
constexpr int kRankCap = 128;   // a threshold digit holding at most this many keys is ranked directly
// queue item types (bits 31:30 of an item code) and extra slot types
constexpr int kItemScore = 0, kItemAttend = 1, kItemComp = 2;
constexpr int kSlotSelect = 3, kSlotMerge = 4, kSlotEnd = 5;
constexpr uint32_t kSpinLimit = 1u << 22;

struct Slot {
  int type, unit, index, L, N, b0, nb, nt, append;
};

// ------------------------------------------------------------------ layout
__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

// scoring item region: kbar rows | Dbar rows | q of the unit (G x D) | the new block's vbar
__host__ __device__ inline int fused_score_bytes(int D, int r, int G) { return kChunk * (D + r) * 4 + G * D * 4 + D * 4; }
__host__ __device__ inline int fused_comp_bytes(int D) { return kChunk2 * D * 4; }
// select scratch: keys | hist | per-warp hist | rank list (key, index) | item factors | bitmap words | word bases
__host__ __device__ inline int fused_select_bytes(int max_cap_blocks, int G) {
  const int nch = (max_cap_blocks + kChunk - 1) / kChunk;
  const int words = align_up((max_cap_blocks + 31) / 32, 4);
  return align_up(max_cap_blocks, 4) * 4 + kBins * 4 + kCW * kPrivBins * 4 + kRankCap * 8 +
         align_up(nch * G, 4) * 4 + 2 * words * 4;
}
__host__ __device__ inline int fused_merge_bytes(int D, int G) { return kCW * G * (D + 2) * 4; }

struct FusedSmem {
  int region[kMaxStages], q, qsq, zs, ss, ws, misc, bars, slots, total;
};

__host__ __device__ inline FusedSmem fused_layout(int D, int r, int G, int region_bytes, int stages) {
  FusedSmem L;
  int off = 0;
  for (int i = 0; i < kMaxStages; ++i) {
    L.region[i] = off;
    if (i < stages) off += region_bytes;
  }
  L.q = off;
  off += G * D * 4;
  L.qsq = off;
  off += align_up(G * r, 4) * 4;
  L.zs = off;
  off += G * kChunk * 4;
  L.ss = off;
  off += G * kChunk * 4;
  L.ws = off;
  off += G * kChunk2 * 4;
  L.misc = off;
  off += 64 * 4;
  L.bars = align_up(off, 16);
  off = L.bars + 2 * kMaxStages * 8;
  L.slots = align_up(off, 16);
  off = L.slots + kMaxStages * (int)sizeof(Slot);
  L.total = align_up(off, 128);
  return L;
}

int fused_region_bytes(int D, int r, int G, int max_cap_blocks) {
  int R = fused_score_bytes(D, r, G);
  const int c = fused_comp_bytes(D), s = fused_select_bytes(max_cap_blocks, G), m = fused_merge_bytes(D, G);
  R = R > c ? R : c;
  R = R > s ? R : s;
  R = R > m ? R : m;
  return align_up(R, 128);
}

int fused_stages(int D, int r, int G, int max_cap_blocks, size_t smem_limit) {
  const int R = fused_region_bytes(D, r, G, max_cap_blocks);
  return (size_t)fused_layout(D, r, G, R, 3).total <= smem_limit ? 3 : 2;
}

size_t fused_smem_bytes(int D, int r, int G, int max_cap_blocks, int stages) {
  return (size_t)fused_layout(D, r, G, fused_region_bytes(D, r, G, max_cap_blocks), stages).total;
}

// misc ints in shared memory
enum Misc { kMFlag = 0, kMCount = 1, kMDigit = 2, kMAbove = 3, kMList = 4, kMBad = 5, kMScan = 8 /* 17 ints */,
            kMLse = 32 /* 8 floats */, kMRef = 40 /* 8 floats */, kMWaitT = 48 /* 2 ints */ };

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Exclusive prefix sum over the consumer threads (one value each).
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
__device__ __forceinline__ int nchunk2(const LayerArgs& a, int s) { return (a.cap_blocks[s] + kChunk2 - 1) / kChunk2; }

// Wait (thread 0, bounded) until `unit` has been selected in this launch;
// returns false on a timeout.  Call with all consumers; it synchronises them.
__device__ __forceinline__ bool wait_ready(const LayerArgs& a, int unit, int* misc) {
  if (threadIdx.x == 0) {
    misc[kMFlag] = 0;
    uint32_t it = 0;
    while (ld_acquire(a.ready + unit) != a.epoch) {
      if (++it > kSpinLimit) {
        set_error(a.status, kDevTimeout, unit / a.Hkv, unit % a.Hkv, 60);
        misc[kMFlag] = 1;
        break;
      }
      __nanosleep(64);
    }
  }
  consumer_sync();
  const bool ok = misc[kMFlag] == 0;
  consumer_sync();
  if (threadIdx.x == 0) reinterpret_cast<unsigned long long*>(misc + kMWaitT)[0] = global_ns();
  return ok;
}

// Optional sub-phase markers for timing studies (compiled in only with
// -DCOMPKV_TRACE_PHASES; they need a trace buffer set with compkv_trace).
#ifdef COMPKV_TRACE_PHASES
#define COMPKV_PHASE(a, id, unit)                                                           \
  do {                                                                                      \
    if (threadIdx.x == 0) {                                                                 \
      const unsigned long long _t = global_ns();                                            \
      trace_record((a), 32 + (id), (unit), 0, _t, _t, _t);                                  \
    }                                                                                       \
  } while (0)
#else
#define COMPKV_PHASE(a, id, unit) \
  do {                            \
  } while (0)
#endif

// ================================================================== producer
template <int D, int G, int MODE>
__device__ void producer(const LayerArgs& a, unsigned char* sm, const FusedSmem& lay, uint64_t* full, uint64_t* empty,
                         Slot* slots) {
  // called by lane 0 of the producer warp only
  constexpr bool APPEND = (MODE & kFAppend) != 0;
  const int S = a.stages;
  int st = 0;
  uint32_t uses[kMaxStages] = {0, 0, 0};
  int pub_type[kMaxStages] = {-1, -1, -1}, pub_unit[kMaxStages] = {0, 0, 0};
  int fq_type[8], fq_unit[8], fq_n = 0;

  // count a finished item; queue the unit's follow-up when it was the last
  auto arrive = [&](int type, int u) {
    if (type != kItemScore && type != kItemAttend && type != kItemComp) return;
    const int s = u / a.Hkv;
    int* ctr;
    int target, follow;
    if (type == kItemScore) {
      ctr = a.s1count + u;
      target = a.nchunk[s];
      follow = kSlotSelect;
    } else {
      ctr = a.mcount + u;
      target = a.splits + nchunk2(a, s);
      follow = kSlotMerge;
    }
    fence_gpu();
    const int old = atomicAdd(ctr, 1);
    if (old == target - 1) {
      *ctr = 0;
      fence_gpu();
      fq_type[fq_n] = follow;
      fq_unit[fq_n] = u;
      ++fq_n;
    }
  };
  auto make_slot = [&](int type, int u, int index) {
    Slot sl{type, u, index, 0, 0, 0, 0, 0, 0};
    if (type == kSlotEnd) return sl;
    const int s = u / a.Hkv;
    bool fits;
    sl.L = unit_tokens(a, s, APPEND, &fits);
    sl.N = ceil_blocks(sl.L);
    if (type == kItemScore || type == kItemComp) {
      const int chunk = type == kItemScore ? kChunk : kChunk2;
      sl.b0 = index * chunk;
      sl.nb = sl.b0 < sl.N ? min(chunk, sl.N - sl.b0) : 0;
      // the open block is rewritten by this launch's append: never bulk-copied
      const bool newest = APPEND && fits && sl.nb > 0 && sl.b0 + sl.nb == sl.N;
      sl.append = (type == kItemScore && newest) ? 1 : 0;
      sl.nt = sl.nb - (newest ? 1 : 0);
    }
    return sl;
  };
  auto publish = [&](const Slot& sl) {
    mbar_wait_bounded(&empty[st], (uses[st] & 1) ^ 1, a.status, sl.unit, -1, 40);
    arrive(pub_type[st], pub_unit[st]);
    pub_type[st] = -1;
    slots[st] = sl;
    unsigned char* region = sm + lay.region[st];
    uint32_t bytes = 0;
    const int s = sl.unit / a.Hkv, h = sl.unit % a.Hkv;
    const bool dbar_bulk = (MODE & kFScore) && ((a.r & 3) == 0);
    if (sl.type == kItemScore && sl.nb > 0)
      bytes = (uint32_t)sl.nt * D * 4u + (dbar_bulk ? (uint32_t)sl.nt * a.r * 4u : 0u) + (uint32_t)G * D * 4u;
    if (sl.type == kItemComp && sl.nt > 0) bytes = (uint32_t)sl.nt * D * 4u;
    mbar_arrive_expect_tx(&full[st], bytes);
    if (bytes) {
      const int64_t row0 = row_of(a, s, h, sl.b0);
      if (sl.type == kItemScore) {
        if (sl.nt > 0) {
          bulk_g2s(region, a.kbar + row0 * D, (uint32_t)sl.nt * D * 4u, &full[st]);
          if (dbar_bulk)
            bulk_g2s(region + kChunk * D * 4, a.dbar + row0 * a.r, (uint32_t)sl.nt * a.r * 4u, &full[st]);
        }
        bulk_g2s(region + kChunk * (D + a.r) * 4, a.q + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D,
                 (uint32_t)G * D * 4u, &full[st]);
      } else {
        bulk_g2s(region, a.vbar + row0 * D, (uint32_t)sl.nt * D * 4u, &full[st]);
      }
    }
    if (sl.type == kItemScore || sl.type == kItemAttend || sl.type == kItemComp) {
      pub_type[st] = sl.type;
      pub_unit[st] = sl.unit;
    }
    uses[st]++;
    st = (st + 1 == S) ? 0 : st + 1;
  };
  // settle the counts of every published item, oldest first
  auto drain = [&]() {
    for (int k = 0; k < S; ++k) {
      const int sk = (st + k) % S;
      if (pub_type[sk] < 0) continue;
      mbar_wait_bounded(&empty[sk], (uses[sk] & 1) ^ 1, a.status, pub_unit[sk], -1, 43);
      arrive(pub_type[sk], pub_unit[sk]);
      pub_type[sk] = -1;
    }
  };
  // a SELECT queued in this ring: no new tickets are claimed until it has run,
  // so the CTA does not sit on other units' items while it selects
  int sel_st = -1;
  uint32_t sel_use = 0;
  auto pop_follow = [&]() {
    const Slot sl = make_slot(fq_type[0], fq_unit[0], 0);
    for (int i = 1; i < fq_n; ++i) {
      fq_type[i - 1] = fq_type[i];
      fq_unit[i - 1] = fq_unit[i];
    }
    --fq_n;
    if (sl.type == kSlotSelect) {
      sel_st = st;
      sel_use = uses[st];
    }
    publish(sl);
  };

  bool drained = false;
  int t = -1;
  for (;;) {
    if (fq_n > 0) {
      pop_follow();
      continue;
    }
    if (sel_st >= 0) {
      mbar_wait_bounded(&empty[sel_st], sel_use & 1, a.status, -1, -1, 44);
      sel_st = -1;
    }
    const unsigned long long tp0 = a.trace ? global_ns() : 0ull;
    if (t < 0) t = atomicAdd(a.ticket, 1);
    if (t >= a.total_items) break;
    const int code = __ldg(a.items + t);
    const int type = (code >> 30) & 3, u = (code >> 18) & 0xfff, index = code & 0x3ffff;
    if (type != kItemScore && !drained) {
      drain();
      drained = true;
      continue;
    }
    publish(make_slot(type, u, index));
    if (a.trace) trace_record(a, 16 + type, u, index, tp0, tp0, global_ns());
    t = -1;
  }
  for (;;) {
    drain();
    if (fq_n == 0) break;
    while (fq_n > 0) pop_follow();
  }
  publish(make_slot(kSlotEnd, 0, 0));
}

// Sum of NVAL values over the LPB lanes of a lane group (LPB a power of two,
// NVAL <= LPB): halving steps exchange half of the values, the remaining
// steps add.  On return the lane holds the total of value index `idx`; lanes
// whose `j` is a multiple of LPB / NVAL hold each index exactly once.
template <int NVAL, int LPB>
__device__ __forceinline__ float transpose_reduce_lanes(float (&v)[NVAL], int j, int& idx) {
  int c = NVAL;
  idx = 0;
#pragma unroll
  for (int off = LPB / 2; off > 0; off >>= 1) {
    if (c > 1) {
      const bool up = (j & off) != 0;
#pragma unroll
      for (int i = 0; i < NVAL / 2; ++i) {
        if (i < c / 2) {
          const float send = up ? v[i] : v[i + c / 2];
          const float keep = up ? v[i + c / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      if (up) idx += c / 2;
      c >>= 1;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return v[0];
}

// ================================================================== S item: scoring
template <int D, int G, int MODE>
__device__ void score_item(const LayerArgs& a, const Slot& sl, unsigned char* region, unsigned char* sm,
                           const FusedSmem& lay) {
  constexpr bool SCORE = (MODE & kFScore) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv;
  const int r = a.r;
  const int L = sl.L, N = sl.N, nb = sl.nb, b0 = sl.b0;
  if (nb == 0) return;
  const int rec = chunk_record(a, s, h, sl.index);
  float* sk = reinterpret_cast<float*>(region);
  float* sd = sk + kChunk * D;
  const float* sq = sd + kChunk * r;  // the unit's queries, staged with the rows
  float* svnew = sd + kChunk * r + G * D;
  float* zs = reinterpret_cast<float*>(sm + lay.zs);
  float* ss = reinterpret_cast<float*>(sm + lay.ss);
  const int64_t row0 = row_of(a, s, h, b0);
  if (SCORE && (r & 3))
    for (int i = tid; i < sl.nt * r; i += kCT) sd[i] = a.dbar[row0 * r + i];
  if (sl.append && warp == 0) {
    // pack the new token and recompute the open block's summary
    constexpr int V = D / 32;
    const int b = N - 1, n = L - kBlock * b;
    const int64_t row = row0 + (nb - 1);
    const __nv_bfloat16* kn = a.k_new + ((int64_t)s * a.Hkv + h) * D;
    const __nv_bfloat16* vn = a.v_new + ((int64_t)s * a.Hkv + h) * D;
    store_bf16_raw<V>(a.k + (row * kBlock + n - 1) * D + lane * V, kn + lane * V);
    store_bf16_raw<V>(a.v + (row * kBlock + n - 1) * D + lane * V, vn + lane * V);
    float* kb = sk + (nb - 1) * D;
    float* db = sd + (nb - 1) * r;
    warp_block_summary<D>(a.k + row * kBlock * D, a.v + row * kBlock * D, n, kn, vn, kb, svnew, db, r, lane);
    __syncwarp();
    for (int i = lane; i < D; i += 32) {
      a.kbar[row * D + i] = kb[i];
      a.vbar[row * D + i] = svnew[i];
    }
    for (int i = lane; i < r; i += 32) a.dbar[row * r + i] = db[i];
  }
  consumer_sync();
  COMPKV_PHASE(a, 1, u);
  // ---- zbar and sigma2, LPB lanes per block, shuffle-reduced.  sigma2 is
  // accumulated per lane as sum_i q_{g,i}^2 Dbar_{t(i)} over the lane's
  // coordinates (the same sum as sum_t Qsq_{g,t} Dbar_t, regrouped).
  {
    constexpr int LPB = (G * D / 16 > 32) ? 32 : 16;
    constexpr int NV = D / LPB;
    constexpr int BPW = 32 / LPB;
    constexpr int RUNS = NV / 4 > 0 ? NV / 4 : 1;  // runs of 4 consecutive coordinates per lane
    const int j = lane % LPB, sub = lane / LPB;
    const int gs = D / r;
    float qr[G][NV];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int c = (NV == 8) ? (i < 4 ? 4 * j + i : D / 2 + 4 * j + (i - 4)) : NV * j + i;
        qr[g][i] = sq[g * D + c];
      }
    // with groups of >= 4 coordinates each run lies in one group: pre-sum q^2 per run
    const bool coarse = gs >= 4 && NV >= 4;
    float qrun[G][RUNS];
    int trun[RUNS];
#pragma unroll
    for (int k = 0; k < RUNS; ++k) {
      const int c0 = (NV == 8) ? (k == 0 ? 4 * j : D / 2 + 4 * j) : NV * j;
      trun[k] = c0 / gs;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 4 && i < NV; ++i) t = fmaf(qr[g][4 * k + i], qr[g][4 * k + i], t);
        qrun[g][k] = t;
      }
    }
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
        if (coarse) {
#pragma unroll
          for (int k = 0; k < RUNS; ++k) {
            const float dv = sd[rb * r + trun[k]];
#pragma unroll
            for (int g = 0; g < G; ++g) sacc[g] = fmaf(qrun[g][k], dv, sacc[g]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            const int c = (NV == 8) ? (i < 4 ? 4 * j + i : D / 2 + 4 * j + (i - 4)) : NV * j + i;
            const float dv = sd[rb * r + c / gs];
#pragma unroll
            for (int g = 0; g < G; ++g) sacc[g] = fmaf(qr[g][i] * qr[g][i], dv, sacc[g]);
          }
        }
      }
      // transposed reduction over the block's LPB lanes: each halving step
      // exchanges half of the values, so 2G values cost ~2G shuffles
      constexpr int NVAL = SCORE ? 2 * G : G;
      float vals[NVAL];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        vals[g] = zacc[g];
        if (SCORE) vals[(G + g) % NVAL] = sacc[g];
      }
      int vidx;
      const float tot = transpose_reduce_lanes<NVAL, LPB>(vals, j, vidx);
      if (valid && (j & ((LPB / NVAL > 0 ? LPB / NVAL : 1) - 1)) == 0) {
        if (vidx < G)
          zs[vidx * kChunk + blk] = tot * InvSqrt<D>::v;
        else
          ss[(vidx - G) * kChunk + blk] = tot / (float)D;
      }
    }
  }
  consumer_sync();
  // ---- per query head: item max and sum of e^a, u per block, max of ln|b| + zbar
  COMPKV_PHASE(a, 3, u);
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
    mc = warp_max(mc);
    float la = 0.f;
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
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int blk = lane + 32 * i;
        a.chunk_z[((int64_t)rec * G + g) * kChunk + blk] = (blk < nb) ? zs[g * kChunk + blk] : 0.f;
      }
    }
    if (lane == 0) {
      float* rg = a.chunk_rec + ((int64_t)rec * G + g) * 4;
      rg[0] = ma;
      rg[1] = la;
      rg[2] = mc;
      rg[3] = 0.f;
    }
  }
}

// ================================================================== SELECT follow-up
// Runs once per unit when its last scoring item is done:
//   1. per query head, from the items' records (max a, sum e^(a - max a),
//      max(ln|b| + zbar)): LSE_g, the factors exp(max a - LSE_g) and the
//      compensation reference M_g = max_b (ln|b| + zbar);
//   2. S_b = sum_g u_{g,b} exp(max a - LSE_g) as uint32 keys (S_b >= 0);
//   3. F = {0, N-2, N-1}, then the K-3 largest keys of blocks 1..N-3 by an
//      MSB-first radix select (digits: bits 30:20, 19:9, 8:0), equal keys by
//      increasing block index; a threshold digit holding <= 128 keys is
//      resolved by ranking them directly;
//   4. the ascending list, the bitmap and the count; the compensation
//      accumulator cleared; the unit published as ready.
// With a caller-given selection (attend mode) steps 2-3 are replaced by
// validating the list and building the bitmap from it.
template <int D, int G, int MODE>
__device__ void follow_select(const LayerArgs& a, const Slot& sl, unsigned char* region, int* misc) {
  constexpr bool SEL = (MODE & kFSelect) != 0;
  constexpr bool COMP = (MODE & kFComp) != 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv;
  const int N = sl.N, K = a.K;
  const int nch = (N + kChunk - 1) / kChunk;
  const int rec0 = chunk_record(a, s, h, 0);
  uint32_t* keys = reinterpret_cast<uint32_t*>(region);
  uint32_t* hist = keys + align_up(a.cap_blocks[s], 4);
  uint32_t* phist = hist + kBins;
  uint32_t* lkey = phist + kCW * kPrivBins;
  int* lidx = reinterpret_cast<int*>(lkey + kRankCap);
  float* fch = reinterpret_cast<float*>(lidx + kRankCap);
  unsigned* words = reinterpret_cast<unsigned*>(fch + align_up(((a.cap_blocks[s] + kChunk - 1) / kChunk) * G, 4));
  int* wbase = reinterpret_cast<int*>(words + align_up((a.cap_blocks[s] + 31) / 32, 4));
  float* lse = reinterpret_cast<float*>(misc + kMLse);
  int* selrow = a.sel + (int64_t)u * K;

  // ---- 1. one float4 record per (item, head); eight items in flight per lane
  if (warp < G) {
    const int g = warp;
    float M = -INFINITY, S = 0.f, MC = -INFINITY;
    float ma_keep[8];  // this lane's first eight items' max a, for the factors below
    for (int c0 = lane; c0 < nch; c0 += 256) {
      float4 rv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + 32 * k;
        rv[k] = c < nch ? __ldcg(reinterpret_cast<const float4*>(a.chunk_rec + ((int64_t)(rec0 + c) * G + g) * 4))
                        : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
      }
      if (c0 == lane) {
#pragma unroll
        for (int k = 0; k < 8; ++k) ma_keep[k] = rv[k].x;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        MC = fmaxf(MC, rv[k].z);
        if (SEL && rv[k].x != -INFINITY) {
          const float mn = fmaxf(M, rv[k].x);
          S = (M == -INFINITY ? 0.f : S * expf(M - mn)) + rv[k].y * expf(rv[k].x - mn);
          M = mn;
        }
      }
    }
    MC = warp_max(MC);
    if (SEL) {
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
      if (lane == 0) lse[g] = lg;
      // factors exp(max a - LSE_g) of this lane's items
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = lane + 32 * k;
        if (c < nch) fch[c * G + g] = expf(ma_keep[k] - lg);
      }
      for (int c = lane + 256; c < nch; c += 32)
        fch[c * G + g] = expf(__ldcg(a.chunk_rec + ((int64_t)(rec0 + c) * G + g) * 4) - lg);
    }
    if (COMP && lane == 0) a.unit_ref[u * G + g] = MC;
  }
  if (COMP)
    for (int i = tid; i < G * (D + 4); i += kCT) a.unit_acc[(int64_t)u * G * (D + 4) + i] = 0.f;
  if (SEL)
    for (int i = tid; i < kCW * kPrivBins; i += kCT) phist[i] = 0;
  if (!SEL && tid == 0) {
    misc[kMCount] = 0;
    misc[kMBad] = 0;
  }
  consumer_sync();
  COMPKV_PHASE(a, 11, u);

  if (!SEL) {
    // ---- caller-given selection: validate, count, bitmap
    unsigned* bm = keys;
    const int words = (N + 31) / 32;
    for (int w = tid; w < words; w += kCT) bm[w] = 0u;
    consumer_sync();
    int cnt = 0, bad = 0;
    for (int i = tid; i < K; i += kCT) {
      const int e = __ldcg(selrow + i);
      const int prev = i > 0 ? __ldcg(selrow + i - 1) : -1;
      const bool ok = e >= 0 && e < N && (i == 0 || (prev >= 0 && prev < e));
      if (ok) {
        atomicOr(&bm[e >> 5], 1u << (e & 31));
        ++cnt;
      }
      bad |= (e >= 0 && !ok) || e < -1;
    }
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (cnt) atomicAdd(misc + kMCount, cnt);
      if (bad) misc[kMBad] = 1;
    }
    consumer_sync();
    if (tid == 0) {
      a.unit_nsel[u] = misc[kMCount];
      if (misc[kMBad]) set_error(a.status, kDevBadSelection, s, h, 61);
    }
    for (int w = tid; w < words; w += kCT) a.bitmap[(int64_t)u * a.bm_words + w] = bm[w];
  } else {
    // ---- 2. S_b keys, several four-block groups in flight per thread
    float* scores = a.scores ? a.scores + (int64_t)u * a.score_stride : nullptr;
    constexpr int QB = G >= 8 ? 1 : (G >= 4 ? 3 : 6);
    for (int q0 = 4 * tid; q0 < N; q0 += 4 * kCT * QB) {
      float4 uu[QB][G];
#pragma unroll
      for (int k = 0; k < QB; ++k) {
        const int b4 = q0 + 4 * kCT * k;
#pragma unroll
        for (int g = 0; g < G; ++g)
          uu[k][g] = b4 < N ? __ldcg(reinterpret_cast<const float4*>(
                                  a.chunk_u + ((int64_t)(rec0 + b4 / kChunk) * G + g) * kChunk + (b4 % kChunk)))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < QB; ++k) {
        const int b4 = q0 + 4 * kCT * k;
        if (b4 >= N) continue;
        const int c = b4 / kChunk;
        float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float f = fch[c * G + g];
          S.x = fmaf(uu[k][g].x, f, S.x);
          S.y = fmaf(uu[k][g].y, f, S.y);
          S.z = fmaf(uu[k][g].z, f, S.z);
          S.w = fmaf(uu[k][g].w, f, S.w);
        }
        const float sv[4] = {fmaxf(S.x, 0.f), fmaxf(S.y, 0.f), fmaxf(S.z, 0.f), fmaxf(S.w, 0.f)};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (b4 + i < N) {
            keys[b4 + i] = __float_as_uint(sv[i]);
            if (scores) scores[b4 + i] = sv[i];
          }
      }
    }
    consumer_sync();
    COMPKV_PHASE(a, 12, u);
    if (N > K) {
      // ---- 3. radix select; bit 31 of a key marks it selected (values are >= +0,
      // bit 31 clear).  Digits: the exponent (bits 30:23, per-warp histograms),
      // then bits 22:12 and 11:0 (shared histogram, few keys left).
      int need = K - 3;
      uint32_t prefix = 0, pmask = 0x80000000u;
      bool done = need == 0;
      const int cand_lo = 1, cand_hi = N - 3;
      for (int level = 0; level < 3 && !done; ++level) {
        const int shift = level == 0 ? 23 : (level == 1 ? 12 : 0);
        const int nbins = level == 0 ? kPrivBins : (level == 1 ? 2048 : 4096);
        const uint32_t dmask = (uint32_t)nbins - 1;
        if (level == 0) {
          uint32_t* mine = phist + warp * kPrivBins;
          for (int b = cand_lo + tid; b <= cand_hi; b += kCT) atomicAdd(&mine[keys[b] >> 23], 1u);
          consumer_sync();
          for (int i = tid; i < kPrivBins; i += kCT) {
            uint32_t t = 0;
#pragma unroll
            for (int w = 0; w < kCW; ++w) t += phist[w * kPrivBins + i];
            hist[i] = t;
          }
        } else {
          for (int i = tid; i < nbins; i += kCT) hist[i] = 0;
          consumer_sync();
          for (int b = cand_lo + tid; b <= cand_hi; b += kCT) {
            const uint32_t key = keys[b];
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
          }
        }
        consumer_sync();
        if (warp == 0) {
          // the digit at which the count of larger-or-equal keys reaches `need`
          const int per = nbins / 32;
          int loc = 0;
          for (int i = 0; i < per; ++i) loc += (int)hist[nbins - 1 - per * lane - i];
          int incl = loc;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int before = incl - loc;
          if (before < need && need <= incl) {
            int run = before;
            for (int i = 0; i < per; ++i) {
              const int bin = nbins - 1 - per * lane - i;
              const int c = (int)hist[bin];
              if (run < need && need <= run + c) {
                misc[kMDigit] = bin;
                misc[kMAbove] = run;
              }
              run += c;
            }
          }
          if (lane == 0) misc[kMList] = 0;
        }
        consumer_sync();
        const uint32_t Dg = (uint32_t)misc[kMDigit];
        const int above = misc[kMAbove];
        const int cntD = (int)hist[Dg];
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
        } else if (cntD <= kRankCap) {
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
          for (int e = tid; e < n; e += kCT) {
            const uint32_t k0 = lkey[e];
            const int i0 = lidx[e];
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
        COMPKV_PHASE(a, 13, u);
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
    } else {
      for (int b = tid; b < N; b += kCT) keys[b] |= 0x80000000u;
    }
    consumer_sync();
    COMPKV_PHASE(a, 14, u);
    // ---- 4. bitmap words by ballot, their prefix counts, then the ascending list
    const int nw = (N + 31) / 32;
    for (int w = warp; w < nw; w += kCW) {
      const int b = 32 * w + lane;
      const unsigned word = __ballot_sync(0xffffffffu, b < N && (keys[b] >> 31));
      if (lane == 0) {
        words[w] = word;
        a.bitmap[(int64_t)u * a.bm_words + w] = word;
      }
    }
    consumer_sync();
    if (warp == 0) {
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
      if (lane == 31) {
        const int want = N < K ? N : K;
        if (incl != want) set_error(a.status, kDevInternal, s, h, 50);
        a.unit_nsel[u] = incl;
      }
    }
    consumer_sync();
    for (int w = warp; w < nw; w += kCW) {
      const unsigned word = words[w];
      if ((word >> lane) & 1u) {
        const int pos = wbase[w] + __popc(word & ((1u << lane) - 1u));
        if (pos < K) selrow[pos] = 32 * w + lane;
      }
    }
    {
      const int want = N < K ? N : K;
      for (int i = want + tid; i < K; i += kCT) selrow[i] = -1;
    }
  }
  // ---- publish: the CTA barrier orders every thread's writes before thread 0's release
  consumer_sync();
  if (tid == 0) {
    fence_gpu();
    st_release(a.ready + u, a.epoch);
  }
}

// ================================================================== A item: exact attention
// Sum of P (16 or 32) values across the warp: lane l ends with the total of
// value index l % P (31 shuffles).
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

template <int V>
__device__ __forceinline__ void load_bf16_cg(const __nv_bfloat16* p, float* f) {
  if (V == 4) {
    const uint2 w = __ldcg(reinterpret_cast<const uint2*>(p));
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    f[0] = x.x; f[1] = x.y; f[2 % V] = y.x; f[3 % V] = y.y;
  } else {
    const unsigned w = __ldcg(reinterpret_cast<const unsigned*>(p));
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    f[0] = x.x; f[1 % V] = x.y;
  }
}

template <int D, int G, int MODE>
__device__ void attend_item(const LayerArgs& a, const Slot& sl, unsigned char* region, int* misc) {
  constexpr int V = D / 32;
  constexpr int TG = G >= 8 ? 2 : ((32 / G) > 16 ? 16 : (32 / G));  // tokens per reduction group
  constexpr int P = TG * G;                                          // 16 or 32 values per group
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv, p = sl.index;
  const int L = sl.L, N = sl.N, K = a.K;
  const bool ok = wait_ready(a, u, misc);
  const int* selrow = a.sel + (int64_t)u * K;

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
  const int my_i = p * kCW + warp;
  int b = -1;
  if (ok && my_i < K) {
    const int e = __ldcg(selrow + my_i);
    const int prev = my_i > 0 ? __ldcg(selrow + my_i - 1) : -1;
    if (e >= 0 && e < N && (my_i == 0 || (prev >= 0 && prev < e))) b = e;
  }
  if (b >= 0) {
    // one block per warp: its 16 keys, then its 16 values, each fetched in one round
    constexpr int W = V / 2;  // 32-bit words of this lane's V bf16 coordinates
    constexpr int NG = kBlock / TG;
    const int n = (b == N - 1) ? L - kBlock * b : kBlock;
    const int64_t row = row_of(a, s, h, b);
    const unsigned* kp = reinterpret_cast<const unsigned*>(a.k + row * kBlock * D + lane * V);
    const unsigned* vp = reinterpret_cast<const unsigned*>(a.v + row * kBlock * D + lane * V);
    unsigned raw[kBlock][W];
#pragma unroll
    for (int j = 0; j < kBlock; ++j) {
      if (W == 2) {
        const uint2 w = __ldcg(reinterpret_cast<const uint2*>(kp + j * (D / 2)));
        raw[j][0] = w.x;
        raw[j][W - 1] = w.y;
      } else {
        raw[j][0] = __ldcg(kp + j * (D / 2));
      }
    }
    // logits: lane holds z of (token jj, head gl) for each group of TG tokens
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
      zl[gi] = transpose_reduce<P>(part, lane);
    }
    // block max per head, weights, denominators
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
    for (int j = 0; j < kBlock; ++j) {
      if (W == 2) {
        const uint2 w = __ldcg(reinterpret_cast<const uint2*>(vp + j * (D / 2)));
        raw[j][0] = w.x;
        raw[j][W - 1] = w.y;
      } else {
        raw[j][0] = __ldcg(vp + j * (D / 2));
      }
    }
#pragma unroll
    for (int gi = 0; gi < NG; ++gi) {
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        float vf[V];
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[gi * TG + t][w]));
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
  float* srec = a.split_rec + ((int64_t)u * a.splits + p) * G * (4 + D);
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
}

// ================================================================== C item: Mean compensation
template <int D, int G, int MODE>
__device__ void comp_item(const LayerArgs& a, const Slot& sl, unsigned char* region, unsigned char* sm,
                          const FusedSmem& lay, int* misc) {
  constexpr int V = D / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv;
  const int L = sl.L, N = sl.N, b0 = sl.b0, nb = sl.nb;
  const bool ok = wait_ready(a, u, misc);
  if (!ok || nb == 0) return;
  if (__ldcg(a.unit_nsel + u) >= N) return;  // every block selected: nothing to compensate
  const float* sv = reinterpret_cast<const float*>(region);
  float* ws = reinterpret_cast<float*>(sm + lay.ws);
  float* ref = reinterpret_cast<float*>(misc + kMRef);
  if (tid < G) ref[tid] = __ldcg(a.unit_ref + u * G + tid);
  consumer_sync();
  // weights w = e^(ln|b| + zbar - M_g) of the unselected blocks, 0 for selected ones
  const unsigned* bm = a.bitmap + (int64_t)u * a.bm_words;
  for (int i = tid; i < G * kChunk2; i += kCT) {
    const int g = i / kChunk2, blk = i % kChunk2;
    float w = 0.f;
    if (blk < nb) {
      const int b = b0 + blk;
      const bool selected = (__ldcg(bm + (b >> 5)) >> (b & 31)) & 1u;
      if (!selected) {
        const int n = (b == N - 1) ? L - kBlock * b : kBlock;
        const int rec = chunk_record(a, s, h, b / kChunk);
        const float z = __ldcg(a.chunk_z + ((int64_t)rec * G + g) * kChunk + (b % kChunk));
        w = expf(ln_n(n) + z - ref[g]);
      }
    }
    ws[g * kChunk2 + blk] = w;
  }
  consumer_sync();
  float acc[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) acc[g][i] = 0.f;
  for (int blk = warp; blk < sl.nt; blk += kCW) {
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
  consumer_sync();
  float* red = reinterpret_cast<float*>(region);  // [kCW][G][D], the staged rows are no longer needed
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < V; ++i) red[(warp * G + g) * D + lane * V + i] = acc[g][i];
  consumer_sync();
  float* ua = a.unit_acc + (int64_t)u * G * (D + 4);
  for (int i = tid; i < G * D; i += kCT) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kCW; ++w) t += red[w * G * D + i];
    atomicAdd(ua + (i / D) * (D + 4) + (i % D), t);
  }
  if (warp < G) {
    float t = 0.f;
    for (int blk = lane; blk < kChunk2; blk += 32) t += ws[warp * kChunk2 + blk];
    t = warp_sum(t);
    if (lane == 0) atomicAdd(ua + warp * (D + 4) + D, t);
  }
}

// ================================================================== MERGE follow-up
template <int D, int G>
__device__ void merge_unit(const LayerArgs& a, const Slot& sl) {
  const int tid = threadIdx.x;
  const int u = sl.unit, s = u / a.Hkv, h = u % a.Hkv;
  const int N = sl.N;
  const bool comp = __ldcg(a.unit_nsel + u) < N;
  const float* recs = a.split_rec + (int64_t)u * a.splits * G * (4 + D);
  const float* ua = a.unit_acc + (int64_t)u * G * (D + 4);
  float* out = a.out + ((int64_t)s * a.Hkv * G + (int64_t)h * G) * D;
  const int rs = G * (4 + D);
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
    if (comp) {
      const float mc = __ldcg(a.unit_ref + u * G + g);
      const float cl = __ldcg(ua + g * (D + 4) + D), ca = __ldcg(ua + g * (D + 4) + col);
      if (mc != -INFINITY) {
        const float mn = fmaxf(M, mc);
        const float fo = (M == -INFINITY) ? 0.f : expf(M - mn);
        const float fn = expf(mc - mn);
        ls = ls * fo + cl * fn;
        as = as * fo + ca * fn;
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
  const FusedSmem lay = fused_layout(D, a.r, G, a.region_bytes, a.stages);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + lay.bars);
  uint64_t* empty = full + kMaxStages;
  Slot* slots = reinterpret_cast<Slot*>(sm + lay.slots);
  int* misc = reinterpret_cast<int*>(sm + lay.misc);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (tid >= kCT) {
    // one thread drives the queue; the rest of its warp waits here for it
    if ((tid & 31) == 0) producer<D, G, MODE>(a, sm, lay, full, empty, slots);
    __syncwarp();
  } else {
    int st = 0;
    uint32_t uses[kMaxStages] = {0, 0, 0};
    for (;;) {
      mbar_wait_bounded(&full[st], uses[st] & 1, a.status, -1, -1, 41);
      const Slot sl = slots[st];
      if (sl.type == kSlotEnd) break;
      unsigned char* region = sm + lay.region[st];
      unsigned long long t_item = 0;
      if (a.trace && tid == 0) {
        t_item = global_ns();
        reinterpret_cast<unsigned long long*>(misc + kMWaitT)[0] = t_item;
      }
      switch (sl.type) {
        case kItemScore:
          score_item<D, G, MODE>(a, sl, region, sm, lay);
          break;
        case kItemAttend:
          if (MODE & kFAttend) attend_item<D, G, MODE>(a, sl, region, misc);
          break;
        case kItemComp:
          if (MODE & kFAttend) comp_item<D, G, MODE>(a, sl, region, sm, lay, misc);
          break;
        case kSlotSelect:
          follow_select<D, G, MODE>(a, sl, region, misc);
          break;
        case kSlotMerge:
          merge_unit<D, G>(a, sl);
          break;
        default:
          break;
      }
      consumer_sync();
      if (tid == 0) {
        mbar_arrive(&empty[st]);
        if (a.trace)
          trace_record(a, sl.type, sl.unit, sl.index, t_item, reinterpret_cast<unsigned long long*>(misc + kMWaitT)[0],
                       global_ns());
      }
      uses[st]++;
      st = (st + 1 == a.stages) ? 0 : st + 1;
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
  const size_t sm = (size_t)fused_layout(D, a.r, G, a.region_bytes, a.stages).total;
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
