// Gate-weighted combine: out[t] = g[t,0] * Y[row_of[t,0]] + g[t,1] * Y[row_of[t,1]] in fp32.
//
// m.nxbn.cn/news/48047 3.3 ("output aggregation": expert outputs summed with their gating
// scores); hnwysp.cn/news/30485 2.2 (a token's two expert outputs weighted like [0.6, 0.4]).
// Slot 0 is multiplied and added first, each product rounded to fp32, then the sum rounded once
// (fp32 addition of two terms is commutative, so the result does not depend on slot order).
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
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    const int r0 = a.row_of[2 * (size_t)t], r1 = a.row_of[2 * (size_t)t + 1];
    const float g0 = a.gate[2 * (size_t)t], g1 = a.gate[2 * (size_t)t + 1];
    const float4* y0 = reinterpret_cast<const float4*>(a.y + (size_t)r0 * a.d);
    const float4* y1 = reinterpret_cast<const float4*>(a.y + (size_t)r1 * a.d);
    for (int i = threadIdx.x; i < nvec; i += kCombineThreads) {
      const float4 u = __ldcs(y0 + i), v = __ldcs(y1 + i);
      float4 o;
      o.x = __fadd_rn(__fmul_rn(g0, u.x), __fmul_rn(g1, v.x));
      o.y = __fadd_rn(__fmul_rn(g0, u.y), __fmul_rn(g1, v.y));
      o.z = __fadd_rn(__fmul_rn(g0, u.z), __fmul_rn(g1, v.z));
      o.w = __fadd_rn(__fmul_rn(g0, u.w), __fmul_rn(g1, v.w));
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
