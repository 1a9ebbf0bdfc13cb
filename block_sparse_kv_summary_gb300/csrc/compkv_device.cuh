// Device-side building blocks of the CompKV decode-step kernels (sm_103a).
//
// The launch-argument struct, the scratch layout shared by the two decode
// kernels, inline-PTX wrappers for mbarriers, 1-D bulk (TMA) copies, thread
// block clusters and distributed shared memory, bounded waits that report
// through the device status word, and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace compkv {

constexpr int kBlock = 16;        // tokens per KV block (CompKV, "전제와 한계": block size 16)
constexpr int kMaxBatch = 64;     // sequences per call (launch arguments hold per-sequence tables)
constexpr int kMaxG = 8;
constexpr int kMaxC = 16;         // CTAs of one unit's cluster in the post kernel

// Device status word codes (mirrors compkv_status).
enum DevErr : int {
  kDevOk = 0,
  kDevCapacity = 3,
  kDevTimeout = 5,
  kDevBadSelection = 6,
  kDevInternal = 7,
};

// Ablation switches of "전제와 한계" (bit set = the ablated variant).
enum Variant : int {
  kVarFirstOrderMass = 1,    // drop the 1/2 sigma2 term from the mass estimate
  kVarNoVarianceFactor = 2,  // S_b = sum_g phat (no external variance factor)
  kVarNoCompensation = 4,    // no Mean compensation: renormalise over the selected blocks
};

// Per-call arguments, passed by value (fits the kernel parameter space).
struct LayerArgs {
  // cache of this layer (row 0 = first row of the layer)
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  float* kbar;
  float* vbar;
  float* dbar;
  int* seq_len;               // [B] of this layer
  // inputs / outputs of the call
  const float* q;             // [B][Hkv*G][d]
  const __nv_bfloat16* k_new; // [B][Hkv][d]
  const __nv_bfloat16* v_new;
  float* out;                 // [B][Hkv*G][d]
  int* sel;                   // [B][Hkv][K]
  float* scores;              // [B][Hkv][score_stride] or null
  int score_stride;
  // shape
  int B, Hkv, G, d, r, K;
  int variant;                // Variant bits
  int P;                      // streaming CTAs of the stream kernel (the work plan's CTA count)
  int Q;                      // leading CTAs of the stream kernel's grid that recompute the open blocks
                              // (grid = Q + P; Q = 0 when the call appends nothing)
  int C;                      // CTAs per unit in the post kernel (one cluster)
  int bpc_max;                // post kernel: blocks of one CTA at most (its shared arrays)
  int rec_cap;                // segment records the scratch holds
  // scratch
  int* status;                // [4]: code, sequence, head, site
  int* arrive;                // [1] post clusters past their reads of seq_len (zero between calls)
  float4* rec;                // [rec_cap][G]: max a, sum e^(a - max a), compensation reference, weight sum
  float* comp;                // [rec_cap][G][d]: compensation numerator relative to its reference
  float* zs;                  // [rows][Gp]: zbar per block and head (Gp = max(G, 4))
  float* ss;                  // [rows][Gp]: sigma2 per block and head
  float* anm;                 // [units][G]: a_g of each unit's open block (this call's token joins it)
  // optional trace of the work items (null: off)
  unsigned long long* trace;
  int trace_cap;
  int64_t layer_row0;            // first row of this layer in the whole cache (tensor-map coordinates)
  int kv_host;                   // the K and V rows live in page-locked host memory (reached over the
                                 // chip-to-chip link): blocks are copied by plain 16-byte copies
  int tmap_ok;                   // tmap_k / tmap_v were built; without them blocks take the plain copies
  // tensor maps of the whole K and V caches: 2-D (d, tokens), boxes of 64 x 16
  // bf16 with the 128-byte swizzle; opaque CUtensorMap objects (kernels that
  // use them take the arguments as a grid constant)
  alignas(64) unsigned long long tmap_k[16];
  alignas(64) unsigned long long tmap_v[16];
  // ragged tables
  int64_t seq_row0[kMaxBatch];   // first row of (s, head 0) relative to the layer
  int cap_blocks[kMaxBatch];     // capacity of sequence s in blocks
  int lens[kMaxBatch];           // prefill lengths (compkv_prefill only)
};

__host__ __device__ inline int pad_g(int G) { return G < 4 ? 4 : G; }

__device__ __forceinline__ int64_t row_of(const LayerArgs& a, int s, int h, int b) {
  return a.seq_row0[s] + (int64_t)h * a.cap_blocks[s] + b;
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
  return t;
}

// ---------------------------------------------------------------- status
__device__ __forceinline__ void set_error(int* status, int code, int s, int h, int site) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = s;
    status[2] = h;
    status[3] = site;
  }
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same with an L2 cache policy (createpolicy), e.g. evict-first for data
// read once, so that it does not push the kernels' code and scratch out of L2.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled tensor copy global -> shared of the box at (x, y) of the tensor map
// at `tmap` (a grid-constant kernel argument), completion on `bar`; `dst` is
// 1024-byte aligned (128-byte swizzle) and x * 2 bytes a multiple of 16.
__device__ __forceinline__ void tma_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the load path (any
// memory the device can load from, host memory included); completion is
// awaited with cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Orders this thread's generic-proxy global writes before later async-proxy
// (bulk copy) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// One test for completion of phase `parity` (no suspend hint: the hardware
// decides how long the thread may sleep before the test returns).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`.  Gives up after kWaitNs of %globaltimer
// (a backstop of kWaitPolls tests bounds it even if the timer stalls), records
// a timeout in the status word and returns false.  A decode step takes tens
// of microseconds, so reaching the limit means a copy never arrived.
constexpr unsigned long long kWaitNs = 50ull * 1000 * 1000;  // 50 ms
constexpr uint32_t kWaitPolls = 1u << 26;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status, int s, int h,
                                                  int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0 && global_ns() - t0 > kWaitNs) break;
  }
  set_error(status, kDevTimeout, s, h, site);
  return false;
}

// After a timeout: give the copies this CTA may still have in flight into
// `bar` a bounded time to land (either phase) before the CTA moves on or exits.
__device__ __forceinline__ void mbar_drain_bounded(uint64_t* bar) {
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, 0u) && mbar_try_wait(bar, 1u)) return;
    if ((i & 31) == 0 && global_ns() - t0 > kWaitNs) return;
  }
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync_all() {
  cluster_arrive();
  cluster_wait();
}
// Address of `p` (this CTA's shared memory) in the shared memory of cluster rank `rank`.
__device__ __forceinline__ uint32_t peer_smem(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_peer_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_peer_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  const uint4 u = ld_peer_u4(addr);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}
__device__ __forceinline__ void st_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_peer_u2(uint32_t addr, uint2 v) {
  asm volatile("st.shared::cluster.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_peer_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void red_peer_add(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// ---------------------------------------------------------------- math helpers
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Merge two online-softmax parts (max, sum of e^(x - max)); -inf max = empty.
__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  l = (m == -INFINITY ? 0.f : l * __expf(m - mn)) + (m2 == -INFINITY ? 0.f : l2 * __expf(m2 - mn));
  m = mn;
}

// bf16 x N -> float x N (N = 2 or 4), from an 8- or 4-byte aligned global
// address, through L2 only (the rows may have been written by the kernel
// before, launched with programmatic dependent launch).
template <int N>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float* f);
template <>
__device__ __forceinline__ void load_bf16<4>(const __nv_bfloat16* p, float* f) {
  uint2 u = __ldcg(reinterpret_cast<const uint2*>(p));
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
template <>
__device__ __forceinline__ void load_bf16<2>(const __nv_bfloat16* p, float* f) {
  uint32_t u = __ldcg(reinterpret_cast<const unsigned int*>(p));
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
  f[0] = a.x; f[1] = a.y;
}
template <int N>
__device__ __forceinline__ void store_bf16_raw(__nv_bfloat16* dst, const __nv_bfloat16* src);
template <>
__device__ __forceinline__ void store_bf16_raw<4>(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint2*>(dst) = __ldcg(reinterpret_cast<const uint2*>(src));
}
template <>
__device__ __forceinline__ void store_bf16_raw<2>(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint32_t*>(dst) = __ldcg(reinterpret_cast<const unsigned int*>(src));
}

__device__ __forceinline__ int ceil_blocks(int L) { return (L + kBlock - 1) / kBlock; }

// ln n for the token count n = 1..16 of a block (the log of |b|), as a table:
// the values are the correctly rounded natural logarithms of the integers.
static __constant__ float c_ln_count[kBlock + 1] = {
    0.f,                 0.f,                 0.6931471805599453f, 1.0986122886681098f, 1.3862943611198906f,
    1.6094379124341003f, 1.791759469228055f,  1.9459101090932196f, 2.0794415416798357f, 2.1972245773362196f,
    2.302585092994046f,  2.3978952727983707f, 2.4849066497880004f, 2.5649493574615367f, 2.6390573296152584f,
    2.70805020110221f,   2.772588722239781f};
__device__ __forceinline__ float ln_count(int n) { return n == kBlock ? 2.772588722239781f : c_ln_count[n]; }

// Tokens of sequence s in this call: the stored length, plus one when the
// call appends and the sequence has room (`fits`).
__device__ __forceinline__ int call_tokens(int Lold, int cap_blocks, bool append, bool* fits) {
  const int cap = cap_blocks * kBlock;
  *fits = Lold >= 0 && Lold < cap;
  int L = Lold < 0 ? 0 : (Lold > cap ? cap : Lold);
  if (append && *fits) L += 1;
  return L;
}

// ---------------------------------------------------------------- work plan
// The stream kernel splits every unit (sequence s, KV head h) of the layer
// into segments of `seg` consecutive blocks (the last one shorter), numbered
// unit by unit: sequence-major, then head, then position.  seg is the
// smallest multiple of `sb` with P segments' worth of blocks covering the
// layer, so there are at most P + units segments.
struct Plan {
  int seg;       // blocks per segment
  int total;     // segments of the layer
};
__device__ __forceinline__ int plan_seg(long long blocks_total, int P, int sb) {
  long long s = (blocks_total + P - 1) / P;
  s = (s + sb - 1) / sb * sb;
  return (int)(s < sb ? sb : s);
}

}  // namespace compkv
