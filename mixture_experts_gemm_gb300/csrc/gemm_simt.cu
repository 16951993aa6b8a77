// fp32 grouped expert GEMM on the SIMT FMA pipes (the fp32 dtype path).
//
// tcgen05 has no fp32-input kind and TF32 (10-bit mantissa) cannot hold fp32 parity, so fp32
// layers run here: one CTA per (expert, 32-row slice of a 128-row tile, 32-column tile), 256
// threads with a 2x2 register tile each (slices past the expert's rows exit at once, so the work
// follows the real row count), K staged through shared memory 32 at a time; the global loads of the next K
// slab are issued into registers before the current slab is multiplied, so their latency overlaps
// the FMAs (these layers are small: latency, not FMA throughput, sets their time).  Each expert is
// an affine layer out = in W^T (+ b) with W stored [out, in] (hnwysp.cn/news/30485 3.2), two layers per expert
// W1 | b1 | W2 | b2 (m.nxbn.cn/news/48047 3.1), the activation applied in the epilogue
// (m.nxbn.cn 2.1: matmul and activation fused per expert).  With two slots and an fp32 output the
// down projection's epilogue also does the combine (m.nxbn.cn 3.3): g * y added onto the cleared
// output row of the row's token.
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int SBM = 32, SBN = 32, SBK = 32;
constexpr int kSlices = kRowTile / SBM;  // row slices per 128-row tile
constexpr int TM = SBM / 16;             // rows per thread
constexpr int TN = SBN / 16;             // columns per thread
constexpr int kLoadsA = SBM * SBK / 256, kLoadsB = SBN * SBK / 256;  // per thread per K slab

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemmArgs a) {
  constexpr bool kSwiGLU = EPI == kEpiSwiGLU;
  __shared__ float As[SBK][SBM + 4];
  __shared__ float Bs[SBK][SBN + 4];
  __shared__ float B3s[kSwiGLU ? SBK : 1][SBN + 4];
  const Sched* sc = a.sched;
  const int n_tiles = (a.N + SBN - 1) / SBN;
  const int tile = blockIdx.x / kSlices, slice = blockIdx.x % kSlices;
  pdl_trigger();
  pdl_wait();
  if (tile >= sc->mtile_start[a.E] * n_tiles) return;
  int e = 0;
  while (e + 1 < a.E && sc->mtile_start[e + 1] * n_tiles <= tile) ++e;
  const int local = tile - sc->mtile_start[e] * n_tiles;
  const int mt_e = sc->mtile_start[e + 1] - sc->mtile_start[e];
  const int n = local / mt_e, m = local - n * mt_e;
  const int row0 = sc->offsets[e] + m * kRowTile + slice * SBM;
  const int seg_end = sc->offsets[e] + sc->counts[e];
  if (row0 >= seg_end) return;  // padding rows only
  const int n0 = n * SBN;
  const float* __restrict__ A = a.a;
  const float* __restrict__ B = a.b + (size_t)e * a.N * a.K;
  const float* __restrict__ B3 = kSwiGLU ? a.b3 + (size_t)e * a.N * a.K : nullptr;

  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[TM][TN], acc3[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = acc3[i][j] = 0.f;

  float ra[kLoadsA], rb[kLoadsB], rb3[kSwiGLU ? kLoadsB : 1];
  auto load_slab = [&](int k0) {
#pragma unroll
    for (int i = 0; i < kLoadsA; ++i) {
      const int id = tid + i * 256, r = id / SBK, k = id % SBK;
      ra[i] = (k0 + k < a.K) ? A[(size_t)(row0 + r) * a.K + k0 + k] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kLoadsB; ++i) {
      const int id = tid + i * 256, c = id / SBK, k = id % SBK;
      const bool in = (n0 + c < a.N) && (k0 + k < a.K);
      rb[i] = in ? B[(size_t)(n0 + c) * a.K + k0 + k] : 0.f;
      if constexpr (kSwiGLU) rb3[i] = in ? B3[(size_t)(n0 + c) * a.K + k0 + k] : 0.f;
    }
  };
  load_slab(0);
  for (int k0 = 0; k0 < a.K; k0 += SBK) {
    __syncthreads();  // every thread is done with the previous slab
#pragma unroll
    for (int i = 0; i < kLoadsA; ++i) {
      const int id = tid + i * 256;
      As[id % SBK][id / SBK] = ra[i];
    }
#pragma unroll
    for (int i = 0; i < kLoadsB; ++i) {
      const int id = tid + i * 256;
      Bs[id % SBK][id / SBK] = rb[i];
      if constexpr (kSwiGLU) B3s[id % SBK][id / SBK] = rb3[i];
    }
    __syncthreads();
    if (k0 + SBK < a.K) load_slab(k0 + SBK);  // in flight while this slab is multiplied
#pragma unroll
    for (int kk = 0; kk < SBK; ++kk) {
      float af[TM], bf[TN], bf3[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) af[i] = As[kk][ty * TM + i];
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        bf[j] = Bs[kk][tx * TN + j];
        if constexpr (kSwiGLU) bf3[j] = B3s[kk][tx * TN + j];
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          acc[i][j] = fmaf(af[i], bf[j], acc[i][j]);
          if constexpr (kSwiGLU) acc3[i][j] = fmaf(af[i], bf3[j], acc3[i][j]);
        }
    }
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = row0 + ty * TM + i;
    if (r >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int col = n0 + tx * TN + j;
      if (col >= a.N) continue;
      float v = acc[i][j];
      if constexpr (EPI == kEpiSwiGLU) {
        v = (v / (1.0f + expf(-v))) * acc3[i][j];
      } else if constexpr (EPI == kEpiReluBias) {
        v = fmaxf(v + a.bias[(size_t)e * a.N + col], 0.f);
      } else {
        if (a.bias) v += a.bias[(size_t)e * a.N + col];
        if (a.comb_out) {  // two slots added onto zero: the sum is the same in either order
          atomicAdd(&a.comb_out[(size_t)a.token_of_row[r] * a.N + col], __fmul_rn(a.gate_of_row[r], v));
          continue;
        }
      }
      a.out[(size_t)r * a.N + col] = v;
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(int epi, const SimtGemmArgs& a, int max_mtiles, cudaStream_t s) {
  const int n_tiles = (a.N + SBN - 1) / SBN;
  const int grid = max_mtiles * n_tiles * kSlices;
  if (grid <= 0) return cudaSuccess;
  switch (epi) {
    case kEpiSwiGLU: return pdl_launch(simt_gemm_kernel<kEpiSwiGLU>, dim3(grid), dim3(256), 0, s, a);
    case kEpiReluBias: return pdl_launch(simt_gemm_kernel<kEpiReluBias>, dim3(grid), dim3(256), 0, s, a);
    default: return pdl_launch(simt_gemm_kernel<kEpiStoreF32>, dim3(grid), dim3(256), 0, s, a);
  }
}

}  // namespace colibri
