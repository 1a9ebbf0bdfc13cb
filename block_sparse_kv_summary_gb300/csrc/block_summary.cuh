// Summary of one 16-token block by one warp (CompKV, section "무엇과 다른가":
// {|b|, kbar_b, Dbar_b, vbar_b}).  Lane l holds D/32 consecutive coordinates
// of every token.  Mean and population variance are two-pass in fp32 from the
// exact bf16 values (mean first, then squared deviations from it), so there
// is no E[k^2] - E[k]^2 cancellation.  Dbar_t is the mean of the variances
// of the contiguous coordinate group t = [t*D/r, (t+1)*D/r).  When `knew` is
// given, token n-1 is taken from knew/vnew instead of the rows.  Outputs are
// generic pointers (global or shared memory).
#pragma once

#include "compkv_device.cuh"

namespace compkv {

template <int D>
__device__ __forceinline__ void warp_block_summary(const __nv_bfloat16* krow, const __nv_bfloat16* vrow, int n,
                                                   const __nv_bfloat16* knew, const __nv_bfloat16* vnew,
                                                   float* kbar, float* vbar, float* dbar, int r, int lane) {
  constexpr int V = D / 32;
  float kt[kBlock][V];
  float ks[V], vs[V];
#pragma unroll
  for (int i = 0; i < V; ++i) ks[i] = vs[i] = 0.f;
#pragma unroll
  for (int j = 0; j < kBlock; ++j) {
    if (j < n) {
      const bool is_new = (knew != nullptr) && (j == n - 1);
      const __nv_bfloat16* kp = is_new ? knew + lane * V : krow + j * D + lane * V;
      const __nv_bfloat16* vp = is_new ? vnew + lane * V : vrow + j * D + lane * V;
      float vf[V];
      load_bf16<V>(kp, kt[j]);
      load_bf16<V>(vp, vf);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        ks[i] += kt[j][i];
        vs[i] += vf[i];
      }
    }
  }
  const float fn = (float)n;
  float mean[V], var[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    mean[i] = ks[i] / fn;
    var[i] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < kBlock; ++j) {
    if (j < n) {
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float dlt = kt[j][i] - mean[i];
        var[i] = fmaf(dlt, dlt, var[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    var[i] = var[i] / fn;
    kbar[lane * V + i] = mean[i];
    vbar[lane * V + i] = vs[i] / fn;
  }
  // grouped mean of the variances: group t = coordinates [t*D/r, (t+1)*D/r)
  const int gs = D / r;
  if (gs >= V) {
    const int lpg = gs / V;  // lanes per group (power of two)
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) t += var[i];
    for (int o = lpg >> 1; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((lane & (lpg - 1)) == 0) dbar[lane / lpg] = t / (float)gs;
  } else {
    const int per = V / gs;  // groups per lane
    for (int t = 0; t < per; ++t) {
      float sum = 0.f;
      for (int c = 0; c < gs; ++c) sum += var[t * gs + c];
      dbar[lane * per + t] = sum / (float)gs;
    }
  }
}

}  // namespace compkv
