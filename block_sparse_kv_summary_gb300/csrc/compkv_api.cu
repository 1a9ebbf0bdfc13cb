// C-ABI entry points of libcompkv.so: argument validation, the scratch layout,
// and the launch sequence of each call.  See include/compkv.h for the contract.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched through the runtime)
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/compkv.h"
#include "compkv_launch.h"

using namespace compkv;

namespace {

thread_local char g_last_error[512] = "";

compkv_status fail(compkv_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

constexpr size_t kMaxSmem = 232448;   // 227 KiB of shared memory per CTA
constexpr size_t kPostSoft = 113 * 1024;  // two post CTAs per multiprocessor (16-CTA clusters co-resident)
constexpr int kBpcLimit = 8192;            // blocks of one post CTA at most

struct Layout {
  std::vector<int> cap_blocks;
  std::vector<int64_t> seq_row0;
  int64_t rows_per_layer = 0;
  int max_cap_blocks = 0;
  int K = 0, C = 0, bpc_max = 0, units = 0, rec_cap = 0;
  size_t off_status = 0, off_arrive = 0, off_rec = 0, off_comp = 0, off_zs = 0, off_ss = 0, off_anm = 0, off_sel = 0,
         off_hq = 0,
         off_hk = 0, off_hv = 0, off_hout = 0, total = 0;
};

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

compkv_status make_layout(const compkv_config* c, Layout* L) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "config is NULL");
  if (c->num_layers < 1) return fail(COMPKV_ERR_INVALID_ARG, "num_layers must be >= 1 (got %d)", c->num_layers);
  if (c->batch < 1 || c->batch > kMaxBatch)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "batch must be in 1..%d (got %d)", kMaxBatch, c->batch);
  if (c->num_kv_heads < 1 || c->num_kv_heads > 32)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "num_kv_heads must be in 1..32 (got %d)", c->num_kv_heads);
  if (!(c->group_size == 1 || c->group_size == 2 || c->group_size == 4 || c->group_size == 8))
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "group_size must be 1, 2, 4 or 8 (got %d)", c->group_size);
  if (!(c->head_dim == 64 || c->head_dim == 128))
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "head_dim must be 64 or 128 (got %d)", c->head_dim);
  if (c->block_size != kBlock) return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "block_size must be 16 (got %d)", c->block_size);
  if (!is_pow2(c->r) || c->r > c->head_dim || c->head_dim % c->r)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "r must be a power of two dividing head_dim (got %d)", c->r);
  if (c->budget_tokens % kBlock || c->budget_tokens / kBlock < 3 || c->budget_tokens / kBlock > 65536)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "budget_tokens must be a multiple of 16 in 48..1048576 (got %d)",
                c->budget_tokens);
  if (c->variant & ~(COMPKV_VARIANT_FIRST_ORDER_MASS | COMPKV_VARIANT_NO_VARIANCE_FACTOR | COMPKV_VARIANT_NO_COMPENSATION))
    return fail(COMPKV_ERR_INVALID_ARG, "variant has unknown bits (got %d)", c->variant);
  L->cap_blocks.resize(c->batch);
  for (int s = 0; s < c->batch; ++s) {
    const int cap = c->capacity_tokens ? c->capacity_tokens[s] : c->max_tokens;
    if (cap < kBlock || cap % kBlock)
      return fail(COMPKV_ERR_INVALID_ARG, "capacity of sequence %d must be a positive multiple of 16 (got %d)", s, cap);
    L->cap_blocks[s] = cap / kBlock;
  }
  const int H = c->num_kv_heads, G = c->group_size, d = c->head_dim;
  L->seq_row0.resize(c->batch);
  int64_t row = 0;
  L->max_cap_blocks = 0;
  for (int s = 0; s < c->batch; ++s) {
    L->seq_row0[s] = row;
    row += (int64_t)H * L->cap_blocks[s];
    if (L->cap_blocks[s] > L->max_cap_blocks) L->max_cap_blocks = L->cap_blocks[s];
  }
  L->rows_per_layer = row;
  L->K = c->budget_tokens / kBlock;
  // the post kernel's cluster: one selected block per warp and round (8 warps), and every CTA's
  // share of a unit's blocks in shared memory; smallest C whose shared memory allows two CTAs
  // per multiprocessor, else the smallest that fits at all
  const int c0 = (L->K + 7) / 8 < 1 ? 1 : ((L->K + 7) / 8 > kMaxC ? kMaxC : (L->K + 7) / 8);
  auto bpc_of = [&](int C) { return ((L->max_cap_blocks + C - 1) / C + 3) & ~3; };
  L->C = 0;
  for (int C = c0; C <= kMaxC && !L->C; ++C)
    if (bpc_of(C) <= kBpcLimit && post_smem(d, G, C, bpc_of(C), L->K) <= kPostSoft) L->C = C;
  for (int C = c0; C <= kMaxC && !L->C; ++C)
    if (bpc_of(C) <= kBpcLimit && post_smem(d, G, C, bpc_of(C), L->K) <= kMaxSmem) L->C = C;
  if (!L->C || stream_smem(d, c->r, G) > kMaxSmem)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE,
                "a sequence capacity of %d blocks does not fit the selection in shared memory", L->max_cap_blocks);
  L->bpc_max = bpc_of(L->C);
  L->units = c->batch * H;
  L->rec_cap = kMaxStreamCtas + L->units;
  const int Gp = pad_g(G);
  size_t off = 0;
  auto region = [&](size_t* o, size_t bytes) {
    *o = off;
    off = round256(off + bytes);
  };
  region(&L->off_status, 16);
  region(&L->off_arrive, 16);
  region(&L->off_rec, (size_t)L->rec_cap * G * 4 * sizeof(float));
  region(&L->off_comp, (size_t)L->rec_cap * G * d * sizeof(float));
  region(&L->off_zs, (size_t)row * Gp * sizeof(float));
  region(&L->off_ss, (size_t)row * Gp * sizeof(float));
  region(&L->off_anm, (size_t)L->units * G * sizeof(float));
  region(&L->off_sel, (size_t)L->units * L->K * sizeof(int));
  // staging of compkv_decode_host: q, k_new, v_new and out of one call
  region(&L->off_hq, (size_t)L->units * G * d * sizeof(float));
  region(&L->off_hk, (size_t)L->units * d * 2);
  region(&L->off_hv, (size_t)L->units * d * 2);
  region(&L->off_hout, (size_t)L->units * G * d * sizeof(float));
  L->total = off;
  return COMPKV_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

struct ProfSlot {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
  double ms = 0.0;
  int64_t count = 0;
};

struct compkv_ctx {
  compkv_config cfg;
  compkv_buffers buf;
  Layout lay;
  CUtensorMap tmap_k, tmap_v;  // the whole K and V caches, for the post kernel's block copies
  int tmap_ok = 0;             // the maps were built
  int kv_host = 0;             // K and V in page-locked host memory (no tensor maps)
  int64_t launches = 0;
  unsigned long long* trace = nullptr;
  int trace_cap = 0;
  int prof = 0;  // 0 off, 1 per call, 2 per call and per kernel of a chain
  ProfSlot slots[COMPKV_KERNEL_FAMILIES];
  std::vector<cudaEvent_t> pool;
  ~compkv_ctx() {
    for (auto& sl : slots)
      for (auto& pr : sl.pending) {
        cudaEventDestroy(pr.first);
        cudaEventDestroy(pr.second);
      }
    for (auto e : pool) cudaEventDestroy(e);
  }
};

namespace {

// Multiprocessors of the current device (queried once per device).
int device_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64) {
    const int v = cached[dev].load();
    if (v > 0) return v;
  }
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n);
  return n;
}

// Stream CTAs of the decode chain on the current device for (d, r, G):
// multiprocessors x resident CTAs, cached per device.
int device_stream_ctas(int d, int r, int G) {
  static std::atomic<int> cache[64][2][8][4];  // [dev][d == 128][log2 r][log2 G]
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kMaxStreamCtas / 4;
  int lr = 0, lg = 0;
  while ((1 << lr) < r) ++lr;
  while ((1 << lg) < G) ++lg;
  std::atomic<int>& slot = cache[dev][d == 128][lr][lg];
  int v = slot.load();
  if (v > 0) return v;
  const int per = stream_ctas_per_sm(d, r, G);
  v = device_sms() * (per < 1 ? 1 : per);
  if (v > kMaxStreamCtas) v = kMaxStreamCtas;
  if (v < 1) v = 1;
  slot.store(v);
  return v;
}

// Tensor maps of the whole K and V caches: 2-D (d, tokens) bf16, boxes of
// 64 x 16 with the 128-byte swizzle (one 16-token block is d / 64 boxes).
compkv_status make_tensor_maps(compkv_ctx* c) {
  // where K and V live: device memory (tensor maps), or page-locked host memory that the device
  // reaches over the chip-to-chip link (plain 16-byte copies, no tensor maps)
  int host = 0;
  for (void* p : {c->buf.k, c->buf.v}) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return fail(COMPKV_ERR_INVALID_ARG, "k / v: not memory the CUDA runtime knows (device or page-locked host)");
    }
    if (at.type == cudaMemoryTypeHost) {
      if (!at.devicePointer || at.devicePointer != p)
        return fail(COMPKV_ERR_INVALID_ARG, "k / v: host memory not mapped at the same address on the device");
      host |= 1 << (p == c->buf.v);
    } else if (at.type != cudaMemoryTypeDevice) {
      return fail(COMPKV_ERR_INVALID_ARG, "k / v must be device memory or page-locked host memory");
    }
  }
  if (host == 1 || host == 2) return fail(COMPKV_ERR_INVALID_ARG, "k and v must both be in device or in host memory");
  c->kv_host = host ? 1 : 0;
  memset(&c->tmap_k, 0, sizeof(c->tmap_k));
  memset(&c->tmap_v, 0, sizeof(c->tmap_v));
  c->tmap_ok = 0;
  if (c->kv_host) return COMPKV_OK;
  static std::atomic<void*> encode_fn{nullptr};
  void* fn = encode_fn.load();
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(COMPKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    encode_fn.store(fn);
  }
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  const int d = c->cfg.head_dim;
  const cuuint64_t tokens = (cuuint64_t)c->cfg.num_layers * (cuuint64_t)c->lay.rows_per_layer * kBlock;
  if (tokens >= (1ull << 31))
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE, "the cache holds %llu token slots; at most 2^31 are addressable",
                (unsigned long long)tokens);
  const cuuint64_t dims[2] = {(cuuint64_t)d, tokens};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {64, kBlock};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap* maps[2] = {&c->tmap_k, &c->tmap_v};
  void* bases[2] = {c->buf.k, c->buf.v};
  for (int i = 0; i < 2; ++i) {
    const CUresult r = reinterpret_cast<Encode>(fn)(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, bases[i], dims,
                                                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(COMPKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  }
  c->tmap_ok = 1;
  return COMPKV_OK;
}

LayerArgs base_args(const compkv_ctx* c, int layer) {
  LayerArgs a;
  memset(&a, 0, sizeof(a));
  static_assert(sizeof(a.tmap_k) == sizeof(CUtensorMap), "tensor map size");
  memcpy(a.tmap_k, &c->tmap_k, sizeof(CUtensorMap));
  memcpy(a.tmap_v, &c->tmap_v, sizeof(CUtensorMap));
  a.layer_row0 = c->lay.rows_per_layer * (int64_t)layer;
  a.kv_host = c->kv_host;
  a.tmap_ok = c->tmap_ok;
  const int d = c->cfg.head_dim, r = c->cfg.r, G = c->cfg.group_size;
  const int64_t rows = c->lay.rows_per_layer * (int64_t)layer;
  a.k = reinterpret_cast<__nv_bfloat16*>(c->buf.k) + rows * kBlock * d;
  a.v = reinterpret_cast<__nv_bfloat16*>(c->buf.v) + rows * kBlock * d;
  a.kbar = c->buf.kbar + rows * d;
  a.vbar = c->buf.vbar + rows * d;
  a.dbar = c->buf.dbar + rows * r;
  a.seq_len = c->buf.seq_len + (int64_t)layer * c->cfg.batch;
  a.B = c->cfg.batch;
  a.Hkv = c->cfg.num_kv_heads;
  a.G = G;
  a.d = d;
  a.r = r;
  a.K = c->lay.K;
  a.variant = c->cfg.variant;
  a.P = device_stream_ctas(d, r, G);
  a.C = c->lay.C;
  a.bpc_max = c->lay.bpc_max;
  a.rec_cap = c->lay.rec_cap;
  char* sc = reinterpret_cast<char*>(c->buf.scratch);
  a.status = reinterpret_cast<int*>(sc + c->lay.off_status);
  a.arrive = reinterpret_cast<int*>(sc + c->lay.off_arrive);
  a.rec = reinterpret_cast<float4*>(sc + c->lay.off_rec);
  a.comp = reinterpret_cast<float*>(sc + c->lay.off_comp);
  a.zs = reinterpret_cast<float*>(sc + c->lay.off_zs);
  a.ss = reinterpret_cast<float*>(sc + c->lay.off_ss);
  a.anm = reinterpret_cast<float*>(sc + c->lay.off_anm);
  a.sel = reinterpret_cast<int*>(sc + c->lay.off_sel);
  a.trace = c->trace;
  a.trace_cap = c->trace_cap;
  for (int s = 0; s < c->cfg.batch; ++s) {
    a.seq_row0[s] = c->lay.seq_row0[s];
    a.cap_blocks[s] = c->lay.cap_blocks[s];
  }
  return a;
}

compkv_status check_call(const compkv_ctx* c, int layer) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  if (layer < 0 || layer >= c->cfg.num_layers)
    return fail(COMPKV_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, c->cfg.num_layers);
  return COMPKV_OK;
}

compkv_status check_ptr(const void* p, const char* name, size_t align) {
  if (!p) return fail(COMPKV_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align)) return fail(COMPKV_ERR_INVALID_ARG, "%s must be %zu-byte aligned", name, align);
  return COMPKV_OK;
}

compkv_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return COMPKV_OK;
  return fail(COMPKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define COMPKV_TRY(x)                    \
  do {                                   \
    compkv_status _st = (x);             \
    if (_st != COMPKV_OK) return _st;    \
  } while (0)

cudaEvent_t take_event(compkv_ctx* c) {
  if (!c->pool.empty()) {
    cudaEvent_t e = c->pool.back();
    c->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launch `kernels` kernels (counted), bracketed by events when profiling is on.
template <class F>
compkv_status launch(compkv_ctx* c, int family, cudaStream_t st, const char* what, F&& fn, int kernels = 1) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (c->prof) {
    e0 = take_event(c);
    e1 = take_event(c);
    if (e0 && e1) cudaEventRecord(e0, st);
  }
  const cudaError_t e = fn();
  if (e != cudaSuccess) {
    if (e0) c->pool.push_back(e0);
    if (e1) c->pool.push_back(e1);
    return cuda_status(e, what);
  }
  if (e0 && e1) {
    cudaEventRecord(e1, st);
    c->slots[family].pending.emplace_back(e0, e1);
  }
  c->launches += kernels;
  return COMPKV_OK;
}

// A decode-step chain: the stream kernel, then the post kernel.  While
// profiling is on (level 2), each kernel is bracketed by its own events too
// (COMPKV_KERNEL_K_STREAM, _K_POST); the whole call goes under `family`.
compkv_status launch_chain(compkv_ctx* c, int family, const LayerArgs& a, int mode, cudaStream_t st, const char* what) {
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  bool kev = c->prof == 2;
  for (int i = 0; i < 4 && kev; ++i) kev = (ev[i] = take_event(c)) != nullptr;
  if (!kev)
    for (int i = 0; i < 4; ++i)
      if (ev[i]) c->pool.push_back(ev[i]);
  const compkv_status r = launch(
      c, family, st, what,
      [&] {
        cudaError_t e;
        if (kev && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return e;
        if ((e = launch_stream(a, mode, st, true)) != cudaSuccess) return e;
        if (kev && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return e;
        if (kev && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return e;
        if ((e = launch_post(a, mode, st)) != cudaSuccess) return e;
        if (kev && (e = cudaEventRecord(ev[3], st)) != cudaSuccess) return e;
        return cudaSuccess;
      },
      2);
  if (kev) {
    if (r == COMPKV_OK) {
      c->slots[COMPKV_KERNEL_K_STREAM].pending.emplace_back(ev[0], ev[1]);
      c->slots[COMPKV_KERNEL_K_POST].pending.emplace_back(ev[2], ev[3]);
    } else {
      for (int i = 0; i < 4; ++i) c->pool.push_back(ev[i]);
    }
  }
  return r;
}

}  // namespace

extern "C" {

int64_t compkv_rows_per_layer(const compkv_config* cfg) {
  Layout L;
  if (make_layout(cfg, &L) != COMPKV_OK) return 0;
  return L.rows_per_layer;
}

size_t compkv_scratch_bytes(const compkv_config* cfg) {
  Layout L;
  if (make_layout(cfg, &L) != COMPKV_OK) return 0;
  return L.total;
}

compkv_status compkv_init(const compkv_config* cfg, const compkv_buffers* bufs, compkv_ctx** out) {
  g_last_error[0] = 0;
  if (!out) return fail(COMPKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Layout L;
  COMPKV_TRY(make_layout(cfg, &L));
  if (!bufs) return fail(COMPKV_ERR_INVALID_ARG, "buffers are NULL");
  COMPKV_TRY(check_ptr(bufs->k, "k", 16));
  COMPKV_TRY(check_ptr(bufs->v, "v", 16));
  COMPKV_TRY(check_ptr(bufs->kbar, "kbar", 16));
  COMPKV_TRY(check_ptr(bufs->vbar, "vbar", 16));
  COMPKV_TRY(check_ptr(bufs->dbar, "dbar", 16));
  COMPKV_TRY(check_ptr(bufs->seq_len, "seq_len", 4));
  COMPKV_TRY(check_ptr(bufs->scratch, "scratch", 256));
  if (bufs->scratch_bytes < L.total)
    return fail(COMPKV_ERR_INVALID_ARG, "scratch_bytes %zu < required %zu", bufs->scratch_bytes, L.total);
  compkv_ctx* c = new (std::nothrow) compkv_ctx();
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "out of host memory");
  c->cfg = *cfg;
  c->cfg.capacity_tokens = nullptr;  // copied into the layout
  c->buf = *bufs;
  c->lay = L;
  {
    const compkv_status st = make_tensor_maps(c);
    if (st != COMPKV_OK) {
      delete c;
      return st;
    }
  }
  // the kernels' shared memory limits and cluster size, once for this configuration
  cudaError_t e = prepare_stream(cfg->head_dim, cfg->r, cfg->group_size);
  if (e == cudaSuccess) e = prepare_post(cfg->head_dim, cfg->group_size, L.C, L.bpc_max, L.K);
  if (e != cudaSuccess) {
    delete c;
    return cuda_status(e, "setting the kernels' attributes");
  }
  e = cudaMemsetAsync(bufs->scratch, 0, L.total, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) {
    delete c;
    return cuda_status(e, "initialising scratch");
  }
  *out = c;
  return COMPKV_OK;
}

compkv_status compkv_row_offset(const compkv_ctx* c, int layer, int seq, int head, int64_t* first_row,
                                int* capacity_blocks) {
  COMPKV_TRY(check_call(c, layer));
  if (seq < 0 || seq >= c->cfg.batch || head < 0 || head >= c->cfg.num_kv_heads)
    return fail(COMPKV_ERR_INVALID_ARG, "sequence %d / head %d out of range", seq, head);
  if (first_row)
    *first_row = c->lay.rows_per_layer * layer + c->lay.seq_row0[seq] + (int64_t)head * c->lay.cap_blocks[seq];
  if (capacity_blocks) *capacity_blocks = c->lay.cap_blocks[seq];
  return COMPKV_OK;
}

compkv_status compkv_prefill(compkv_ctx* c, int layer, const int* lens, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  if (!lens) return fail(COMPKV_ERR_INVALID_ARG, "lens is NULL");
  LayerArgs a = base_args(c, layer);
  for (int s = 0; s < c->cfg.batch; ++s) {
    if (lens[s] < 0 || lens[s] > c->lay.cap_blocks[s] * kBlock)
      return fail(COMPKV_ERR_CAPACITY, "lens[%d] = %d outside [0, %d]", s, lens[s], c->lay.cap_blocks[s] * kBlock);
    a.lens[s] = lens[s];
  }
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(launch(c, COMPKV_KERNEL_PREFILL, st, "prefill launch",
                    [&] { return launch_prefill(a, c->lay.rows_per_layer, st); }));
  return COMPKV_OK;
}

compkv_status compkv_append(compkv_ctx* c, int layer, const void* k_new, const void* v_new, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  COMPKV_TRY(check_ptr(k_new, "k_new", 16));
  COMPKV_TRY(check_ptr(v_new, "v_new", 16));
  LayerArgs a = base_args(c, layer);
  a.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
  a.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(launch(c, COMPKV_KERNEL_APPEND, st, "append launch", [&] { return launch_append(a, st); }));
  return COMPKV_OK;
}

compkv_status compkv_score_select(compkv_ctx* c, int layer, const float* q, int* sel, float* scores, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  COMPKV_TRY(check_ptr(q, "q", 16));
  COMPKV_TRY(check_ptr(sel, "sel", 16));
  if (scores) COMPKV_TRY(check_ptr(scores, "scores", 16));
  LayerArgs a = base_args(c, layer);
  a.q = q;
  a.sel = sel;
  a.scores = scores;
  a.score_stride = c->lay.max_cap_blocks;
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(launch_chain(c, COMPKV_KERNEL_SCORE, a, kFusedScoreSelect, st, "score/select launch"));
  return COMPKV_OK;
}

compkv_status compkv_attend(compkv_ctx* c, int layer, const float* q, const int* sel, float* out, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  COMPKV_TRY(check_ptr(q, "q", 16));
  COMPKV_TRY(check_ptr(sel, "sel", 16));
  COMPKV_TRY(check_ptr(out, "out", 16));
  LayerArgs a = base_args(c, layer);
  a.q = q;
  a.sel = const_cast<int*>(sel);
  a.out = out;
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(launch_chain(c, COMPKV_KERNEL_ATTEND, a, kFusedAttend, st, "attend launch"));
  return COMPKV_OK;
}

compkv_status compkv_decode(compkv_ctx* c, int layer, const float* q, const void* k_new, const void* v_new, float* out,
                            int* sel, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  COMPKV_TRY(check_ptr(q, "q", 16));
  COMPKV_TRY(check_ptr(k_new, "k_new", 16));
  COMPKV_TRY(check_ptr(v_new, "v_new", 16));
  COMPKV_TRY(check_ptr(out, "out", 16));
  if (sel) COMPKV_TRY(check_ptr(sel, "sel", 16));
  LayerArgs a = base_args(c, layer);
  a.q = q;
  a.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
  a.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
  a.out = out;
  if (sel) a.sel = sel;
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(launch_chain(c, COMPKV_KERNEL_DECODE, a, kFusedDecode, st, "decode launch"));
  return COMPKV_OK;
}

compkv_status compkv_decode_host(compkv_ctx* c, int layer, const float* q_host, const void* k_new_host,
                                 const void* v_new_host, float* out_host, int* sel_host, void* stream) {
  COMPKV_TRY(check_call(c, layer));
  if (!q_host || !k_new_host || !v_new_host || !out_host)
    return fail(COMPKV_ERR_INVALID_ARG, "q, k_new, v_new and out must not be NULL");
  cudaStream_t st = (cudaStream_t)stream;
  char* sc = reinterpret_cast<char*>(c->buf.scratch);
  const size_t units = (size_t)c->lay.units, d = (size_t)c->cfg.head_dim, G = (size_t)c->cfg.group_size;
  float* dq = reinterpret_cast<float*>(sc + c->lay.off_hq);
  void* dk = sc + c->lay.off_hk;
  void* dv = sc + c->lay.off_hv;
  float* dout = reinterpret_cast<float*>(sc + c->lay.off_hout);
  const size_t qb = units * G * d * 4, kb = units * d * 2;
  LayerArgs a = base_args(c, layer);
  a.q = dq;
  a.k_new = reinterpret_cast<const __nv_bfloat16*>(dk);
  a.v_new = reinterpret_cast<const __nv_bfloat16*>(dv);
  a.out = dout;
  // page-locked host buffers (mapped at the same address on the device, 16-byte aligned): the
  // inputs come in through one small kernel and the kernels write out and the selection straight
  // into host memory; any other host memory goes through copies
  // (checked on every call: a buffer freed and its address reused by pageable memory must not
  // be written by a kernel)
  auto mapped = [](const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == p && aligned(p, 16);
  };
  const bool direct = mapped(q_host) && mapped(k_new_host) && mapped(v_new_host) && mapped(out_host) &&
                      (!sel_host || mapped(sel_host)) && qb % 16 == 0 && kb % 16 == 0;
  if (direct) {
    COMPKV_TRY(cuda_status(launch_stage_in(dq, q_host, qb, dk, k_new_host, kb, dv, v_new_host, kb, st), "input stage"));
    ++c->launches;
    a.out = out_host;
    if (sel_host) a.sel = sel_host;
    COMPKV_TRY(launch_chain(c, COMPKV_KERNEL_DECODE, a, kFusedDecode, st, "decode launch"));
  } else {
    COMPKV_TRY(cuda_status(cudaMemcpyAsync(dq, q_host, qb, cudaMemcpyHostToDevice, st), "q copy"));
    COMPKV_TRY(cuda_status(cudaMemcpyAsync(dk, k_new_host, kb, cudaMemcpyHostToDevice, st), "k_new copy"));
    COMPKV_TRY(cuda_status(cudaMemcpyAsync(dv, v_new_host, kb, cudaMemcpyHostToDevice, st), "v_new copy"));
    COMPKV_TRY(launch_chain(c, COMPKV_KERNEL_DECODE, a, kFusedDecode, st, "decode launch"));
    COMPKV_TRY(cuda_status(cudaMemcpyAsync(out_host, dout, qb, cudaMemcpyDeviceToHost, st), "out copy"));
    if (sel_host)
      COMPKV_TRY(cuda_status(cudaMemcpyAsync(sel_host, a.sel, units * (size_t)c->lay.K * 4, cudaMemcpyDeviceToHost, st),
                             "sel copy"));
  }
  COMPKV_TRY(cuda_status(cudaStreamSynchronize(st), "stream synchronize"));
  return COMPKV_OK;
}

compkv_status compkv_device_status(compkv_ctx* c, void* stream) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(cuda_status(cudaStreamSynchronize(st), "stream synchronize"));
  int h[4] = {0, 0, 0, 0};
  int* dev = reinterpret_cast<int*>(reinterpret_cast<char*>(c->buf.scratch) + c->lay.off_status);
  COMPKV_TRY(cuda_status(cudaMemcpyAsync(h, dev, sizeof(h), cudaMemcpyDeviceToHost, st), "status read"));
  COMPKV_TRY(cuda_status(cudaStreamSynchronize(st), "stream synchronize"));
  if (h[0] == 0) return COMPKV_OK;
  COMPKV_TRY(cuda_status(cudaMemsetAsync(dev, 0, sizeof(h), st), "status clear"));
  COMPKV_TRY(cuda_status(cudaStreamSynchronize(st), "stream synchronize"));
  return fail((compkv_status)h[0], "device status %d (sequence %d, head %d, site %d)", h[0], h[1], h[2], h[3]);
}

int64_t compkv_launch_count(const compkv_ctx* c) { return c ? c->launches : 0; }

compkv_status compkv_selftest_wait_timeout(compkv_ctx* c, void* stream) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  cudaStream_t st = (cudaStream_t)stream;
  int* dev = reinterpret_cast<int*>(reinterpret_cast<char*>(c->buf.scratch) + c->lay.off_status);
  COMPKV_TRY(cuda_status(launch_wait_selftest(dev, st), "wait self-test launch"));
  c->launches += 1;
  return COMPKV_OK;
}

compkv_status compkv_trace(compkv_ctx* c, void* buf, size_t bytes) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  if (!buf) {
    c->trace = nullptr;
    c->trace_cap = 0;
    return COMPKV_OK;
  }
  COMPKV_TRY(check_ptr(buf, "trace buffer", 8));
  const size_t header = 8;
  if (bytes < header + 64) return fail(COMPKV_ERR_INVALID_ARG, "trace buffer of %zu bytes holds no record", bytes);
  c->trace = reinterpret_cast<unsigned long long*>(buf);
  const size_t cap = (bytes - header) / 64;
  c->trace_cap = cap > 0x7fffffff ? 0x7fffffff : (int)cap;
  return COMPKV_OK;
}

compkv_status compkv_profile_enable(compkv_ctx* c, int enable) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  if (enable < 0 || enable > 2) return fail(COMPKV_ERR_INVALID_ARG, "profile level %d not in 0..2", enable);
  c->prof = enable;
  return COMPKV_OK;
}

compkv_status compkv_profile_read(compkv_ctx* c, int family, double* total_ms, int64_t* launches) {
  if (!c) return fail(COMPKV_ERR_INVALID_ARG, "context is NULL");
  if (family < 0 || family >= COMPKV_KERNEL_FAMILIES) return fail(COMPKV_ERR_INVALID_ARG, "bad kernel family %d", family);
  ProfSlot& sl = c->slots[family];
  for (auto& pr : sl.pending) {
    COMPKV_TRY(cuda_status(cudaEventSynchronize(pr.second), "event synchronize"));
    float ms = 0.f;
    COMPKV_TRY(cuda_status(cudaEventElapsedTime(&ms, pr.first, pr.second), "event elapsed"));
    sl.ms += ms;
    sl.count += 1;
    c->pool.push_back(pr.first);
    c->pool.push_back(pr.second);
  }
  sl.pending.clear();
  if (total_ms) *total_ms = sl.ms;
  if (launches) *launches = sl.count;
  sl.ms = 0.0;
  sl.count = 0;
  return COMPKV_OK;
}

const char* compkv_last_error(void) { return g_last_error; }

const char* compkv_status_string(compkv_status s) {
  switch (s) {
    case COMPKV_OK: return "COMPKV_OK";
    case COMPKV_ERR_INVALID_ARG: return "COMPKV_ERR_INVALID_ARG";
    case COMPKV_ERR_UNSUPPORTED_SHAPE: return "COMPKV_ERR_UNSUPPORTED_SHAPE";
    case COMPKV_ERR_CAPACITY: return "COMPKV_ERR_CAPACITY";
    case COMPKV_ERR_CUDA: return "COMPKV_ERR_CUDA";
    case COMPKV_ERR_TIMEOUT: return "COMPKV_ERR_TIMEOUT";
    case COMPKV_ERR_BAD_SELECTION: return "COMPKV_ERR_BAD_SELECTION";
    case COMPKV_ERR_INTERNAL: return "COMPKV_ERR_INTERNAL";
  }
  return "COMPKV_UNKNOWN";
}

void compkv_destroy(compkv_ctx* c) { delete c; }

}  // extern "C"

// Records `what: detail` as this thread's last error (for other translation units).
compkv_status compkv_internal_fail(compkv_status st, const char* what, const char* detail) {
  return fail(st, "%s: %s", what, detail);
}

// Decode step with a scratch buffer supplied by the caller of this function
// instead of by a context: used by the scratch-free entry point
// (static_scratch.cu).  The status word and counters at the start of the
// scratch are zeroed on `stream` before the launches, so consecutive calls
// that share the buffer start clean.
compkv_status compkv_internal_decode_in(const compkv_config* cfg, const compkv_buffers* bufs, void* scratch,
                                        size_t scratch_bytes, int layer, const float* q, const void* k_new,
                                        const void* v_new, float* out, int* sel, void* stream) {
  g_last_error[0] = 0;
  Layout L;
  COMPKV_TRY(make_layout(cfg, &L));
  if (L.total > scratch_bytes)
    return fail(COMPKV_ERR_UNSUPPORTED_SHAPE,
                "this configuration needs %zu bytes of scratch; the library's static scratch holds %zu", L.total,
                scratch_bytes);
  if (!bufs) return fail(COMPKV_ERR_INVALID_ARG, "buffers are NULL");
  if (layer < 0 || layer >= cfg->num_layers)
    return fail(COMPKV_ERR_INVALID_ARG, "layer %d out of range [0, %d)", layer, cfg->num_layers);
  COMPKV_TRY(check_ptr(bufs->k, "k", 16));
  COMPKV_TRY(check_ptr(bufs->v, "v", 16));
  COMPKV_TRY(check_ptr(bufs->kbar, "kbar", 16));
  COMPKV_TRY(check_ptr(bufs->vbar, "vbar", 16));
  COMPKV_TRY(check_ptr(bufs->dbar, "dbar", 16));
  COMPKV_TRY(check_ptr(bufs->seq_len, "seq_len", 4));
  COMPKV_TRY(check_ptr(scratch, "scratch", 256));
  COMPKV_TRY(check_ptr(q, "q", 16));
  COMPKV_TRY(check_ptr(k_new, "k_new", 16));
  COMPKV_TRY(check_ptr(v_new, "v_new", 16));
  COMPKV_TRY(check_ptr(out, "out", 16));
  if (sel) COMPKV_TRY(check_ptr(sel, "sel", 16));
  compkv_ctx c;
  c.cfg = *cfg;
  c.cfg.capacity_tokens = nullptr;
  c.buf = *bufs;
  c.buf.scratch = scratch;
  c.buf.scratch_bytes = scratch_bytes;
  c.lay = L;
  COMPKV_TRY(make_tensor_maps(&c));
  // no context was initialised for this configuration: the kernels' attributes on every call
  // (queries, and a set only where a limit is still too low)
  cudaError_t ea = prepare_stream(cfg->head_dim, cfg->r, cfg->group_size);
  if (ea == cudaSuccess) ea = prepare_post(cfg->head_dim, cfg->group_size, L.C, L.bpc_max, L.K);
  COMPKV_TRY(cuda_status(ea, "setting the kernels' attributes"));
  cudaStream_t st = (cudaStream_t)stream;
  COMPKV_TRY(cuda_status(cudaMemsetAsync(scratch, 0, L.off_rec, st), "clearing scratch"));
  LayerArgs a = base_args(&c, layer);
  a.q = q;
  a.k_new = reinterpret_cast<const __nv_bfloat16*>(k_new);
  a.v_new = reinterpret_cast<const __nv_bfloat16*>(v_new);
  a.out = out;
  if (sel) a.sel = sel;
  cudaError_t e = launch_stream(a, kFusedDecode, st, true);
  if (e == cudaSuccess) e = launch_post(a, kFusedDecode, st);
  COMPKV_TRY(cuda_status(e, "decode launch"));
  return COMPKV_OK;
}
