// Gate-weighted combine: out[t] = sum over the token's slots s of g[t,s] * Y[row_of[t,s]] in fp32
// (k routed experts, then the shared expert with gate 1 when the layer has one).
//
// m.nxbn.cn/news/48047 3.3 ("output aggregation": expert outputs summed with their gating
// scores); hnwysp.cn/news/30485 2.2 (a token's two expert outputs weighted like [0.6, 0.4]).
// Slots are accumulated in order, each product and each partial sum rounded to fp32 (for two slots
// the result is g0*y0 + g1*y1 rounded once, independent of order).
//
// HBM-bound: per token 2 * d * 4 bytes read, d * sizeof(out) written; float4 loads, coalesced
// 16-byte (fp32) or 8-byte (bf16) stores; one CTA per token row, grid-strided.
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int kCombineThreads = 256;

template <bool kBf16Out>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineArgs a) {
  const int nvec = a.d / 4;
  pdl_trigger();
  pdl_wait();
  const int S = a.S;
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    int r[kMaxSlots];
    float g[kMaxSlots];
#pragma unroll
    for (int s = 0; s < kMaxSlots; ++s) {
      r[s] = s < S ? a.row_of[(size_t)S * t + s] : 0;
      g[s] = s < S ? a.gate[(size_t)S * t + s] : 0.f;
    }
    for (int i = threadIdx.x; i < nvec; i += kCombineThreads) {
      // slot order: o = g0*y0, then o += g_s*y_s; each product and each sum rounded once in fp32
      const float4 u = __ldcs(reinterpret_cast<const float4*>(a.y + (size_t)r[0] * a.d) + i);
      float4 o = make_float4(__fmul_rn(g[0], u.x), __fmul_rn(g[0], u.y), __fmul_rn(g[0], u.z), __fmul_rn(g[0], u.w));
#pragma unroll
      for (int s = 1; s < kMaxSlots; ++s) {
        if (s < S) {
          const float4 v = __ldcs(reinterpret_cast<const float4*>(a.y + (size_t)r[s] * a.d) + i);
          o.x = __fadd_rn(o.x, __fmul_rn(g[s], v.x));
          o.y = __fadd_rn(o.y, __fmul_rn(g[s], v.y));
          o.z = __fadd_rn(o.z, __fmul_rn(g[s], v.z));
          o.w = __fadd_rn(o.w, __fmul_rn(g[s], v.w));
        }
      }
      if constexpr (kBf16Out) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
        uint2 p;
        p.x = *reinterpret_cast<uint32_t*>(&lo);
        p.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (size_t)t * a.d)[i] = p;
      } else {
        reinterpret_cast<float4*>(static_cast<float*>(a.out) + (size_t)t * a.d)[i] = o;
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(int out_dtype, const CombineArgs& a, int num_sms, cudaStream_t s) {
  const int grid = a.T < num_sms * 8 ? a.T : num_sms * 8;
  if (out_dtype == 0) return pdl_launch(combine_kernel<false>, dim3(grid), dim3(kCombineThreads), 0, s, a);
  return pdl_launch(combine_kernel<true>, dim3(grid), dim3(kCombineThreads), 0, s, a);
}

}  // namespace colibri
