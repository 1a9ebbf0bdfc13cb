// Device-side building blocks of the CompKV decode-step kernels (sm_103a).
//
// The launch-argument struct, the scratch record layout, inline-PTX wrappers
// for mbarriers and 1-D bulk (TMA) copies into shared memory, bounded waits
// that report through the device status word, and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace compkv {

constexpr int kBlock = 16;        // tokens per KV block (CompKV, "전제와 한계": block size 16)
constexpr int kMaxBatch = 64;     // sequences per call (launch arguments hold per-sequence tables)
constexpr int kChunk = 64;        // blocks per scoring work item (and per scoring record)
constexpr int kMaxG = 8;

// Device status word codes (mirrors compkv_status).
enum DevErr : int {
  kDevOk = 0,
  kDevCapacity = 3,
  kDevTimeout = 5,
  kDevBadSelection = 6,
  kDevInternal = 7,
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
  int splits;                 // attention CTAs per unit (one cluster)
  // scratch
  int* status;                // [4]: code, sequence, head, site
  int* lnew;                  // [B] tokens of each sequence in this call (after its append)
  float* chunk_rec;           // [chunk records][G][4]: max a, sum e^(a - max a), max(ln|b| + zbar), -
  float* chunk_z;             // [chunk records][G][kChunk]  zbar per block
  float* chunk_s;             // [chunk records][G][kChunk]  sigma2 per block
  float* comp_part;           // [chunk records][G][d + 4]: the chunk's sums with w relative to its own max
  int* unit_nsel;             // [units] selected blocks
  uint32_t* skeys;            // [units][key_stride] S_b as order-preserving keys (full radix selection only)
  int key_stride;             // max capacity in blocks, rounded up to a multiple of 4
  unsigned* hist12;           // [units][4096] histogram of the keys' top 12 bits (full radix selection only)
  int total_chunks;           // scoring items of the layer (64 blocks)
  int sms;                    // multiprocessors of the device
  int post_cpc;               // scoring items owned by one CTA of a unit's cluster (max over sequences)
  // optional trace of the work items (null: off)
  unsigned long long* trace;  // see compkv_trace
  int trace_cap;
  // ragged tables
  int64_t seq_row0[kMaxBatch];   // first row of (s, head 0) relative to the layer
  int cap_blocks[kMaxBatch];     // capacity of sequence s in blocks
  int chunk0[kMaxBatch];         // first chunk record of (s, head 0)
  int nchunk[kMaxBatch];         // chunk records per (s, head) = ceil(cap / kChunk)
  int lens[kMaxBatch];           // prefill lengths (compkv_prefill only)
};

__device__ __forceinline__ int64_t row_of(const LayerArgs& a, int s, int h, int b) {
  return a.seq_row0[s] + (int64_t)h * a.cap_blocks[s] + b;
}

// ---------------------------------------------------------------- tracing
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
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

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Test for completion of phase `parity`; a waiting thread is suspended (it
// issues nothing) until the phase completes or about kSuspendNs pass.
constexpr uint32_t kSuspendNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`; gives up after a bounded number of polls
// (a few seconds at most), records a timeout in the status word and returns
// false.
constexpr uint32_t kWaitPolls = 1u << 12;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status, int s, int h,
                                                  int site) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_error(status, kDevTimeout, s, h, site);
  // give copies still in flight a second bounded chance to land before the CTA exits
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait(bar, parity)) break;
  return false;
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

// bf16 x N -> float x N (N = 2 or 4), from an 8- or 4-byte aligned address.
template <int N>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float* f);
template <>
__device__ __forceinline__ void load_bf16<4>(const __nv_bfloat16* p, float* f) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
template <>
__device__ __forceinline__ void load_bf16<2>(const __nv_bfloat16* p, float* f) {
  uint32_t u = *reinterpret_cast<const uint32_t*>(p);
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
  f[0] = a.x; f[1] = a.y;
}
template <int N>
__device__ __forceinline__ void store_bf16_raw(__nv_bfloat16* dst, const __nv_bfloat16* src);
template <>
__device__ __forceinline__ void store_bf16_raw<4>(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
}
template <>
__device__ __forceinline__ void store_bf16_raw<2>(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
}

__device__ __forceinline__ int ceil_blocks(int L) { return (L + kBlock - 1) / kBlock; }

}  // namespace compkv
