// fp32 grouped expert GEMM on the SIMT FMA pipes (the fp32 dtype path).
//
// tcgen05 has no fp32-input kind and TF32 (10-bit mantissa) cannot hold fp32 parity, so fp32
// layers run here: one CTA per (expert, 128-row tile, 64-column tile), 256 threads with an 8x4
// register tile each, K staged through shared memory 16 at a time.  Each expert is an affine layer
// out = in W^T (+ b) with W stored [out, in] (hnwysp.cn/news/30485 3.2), two layers per expert
// W1 | b1 | W2 | b2 (m.nxbn.cn/news/48047 3.1), the activation applied in the epilogue
// (m.nxbn.cn 2.1: matmul and activation fused per expert).
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int SBM = 128, SBN = 64, SBK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemmArgs a) {
  constexpr bool kSwiGLU = EPI == kEpiSwiGLU;
  __shared__ float As[SBK][SBM + 4];
  __shared__ float Bs[SBK][SBN + 4];
  __shared__ float B3s[kSwiGLU ? SBK : 1][SBN + 4];
  const Sched* sc = a.sched;
  const int n_tiles = (a.N + SBN - 1) / SBN;
  const int tile = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (tile >= sc->mtile_start[a.E] * n_tiles) return;
  int e = 0;
  while (e + 1 < a.E && sc->mtile_start[e + 1] * n_tiles <= tile) ++e;
  const int local = tile - sc->mtile_start[e] * n_tiles;
  const int mt_e = sc->mtile_start[e + 1] - sc->mtile_start[e];
  const int n = local / mt_e, m = local - n * mt_e;
  const int row0 = sc->offsets[e] + m * SBM;
  const int seg_end = sc->offsets[e] + sc->counts[e];
  const int n0 = n * SBN;
  const float* __restrict__ A = a.a;
  const float* __restrict__ B = a.b + (size_t)e * a.N * a.K;
  const float* __restrict__ B3 = kSwiGLU ? a.b3 + (size_t)e * a.N * a.K : nullptr;

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[8][4], acc3[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = acc3[i][j] = 0.f;

  for (int k0 = 0; k0 < a.K; k0 += SBK) {
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int id = tid + i * 256, r = id >> 4, k = id & 15;
      As[k][r] = (k0 + k < a.K) ? A[(size_t)(row0 + r) * a.K + k0 + k] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int id = tid + i * 256, c = id >> 4, k = id & 15;
      const bool in = (n0 + c < a.N) && (k0 + k < a.K);
      Bs[k][c] = in ? B[(size_t)(n0 + c) * a.K + k0 + k] : 0.f;
      if constexpr (kSwiGLU) B3s[k][c] = in ? B3[(size_t)(n0 + c) * a.K + k0 + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      float af[8], bf[4], bf3[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) af[i] = As[kk][ty * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bf[j] = Bs[kk][tx * 4 + j];
        if constexpr (kSwiGLU) bf3[j] = B3s[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
          if constexpr (kSwiGLU) acc3[i][j] = fmaf(af[i], bf3[j], acc3[i][j]);
        }
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = row0 + ty * 8 + i;
    if (r >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= a.N) continue;
      float v = acc[i][j];
      if constexpr (EPI == kEpiSwiGLU) {
        v = (v / (1.0f + expf(-v))) * acc3[i][j];
      } else if constexpr (EPI == kEpiReluBias) {
        v = fmaxf(v + a.bias[(size_t)e * a.N + col], 0.f);
      } else {
        if (a.bias) v += a.bias[(size_t)e * a.N + col];
      }
      a.out[(size_t)r * a.N + col] = v;
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(int epi, const SimtGemmArgs& a, int max_mtiles, cudaStream_t s) {
  const int n_tiles = (a.N + SBN - 1) / SBN;
  const int grid = max_mtiles * n_tiles;
  if (grid <= 0) return cudaSuccess;
  switch (epi) {
    case kEpiSwiGLU: return pdl_launch(simt_gemm_kernel<kEpiSwiGLU>, dim3(grid), dim3(256), 0, s, a);
    case kEpiReluBias: return pdl_launch(simt_gemm_kernel<kEpiReluBias>, dim3(grid), dim3(256), 0, s, a);
    default: return pdl_launch(simt_gemm_kernel<kEpiStoreF32>, dim3(grid), dim3(256), 0, s, a);
  }
}

}  // namespace colibri
