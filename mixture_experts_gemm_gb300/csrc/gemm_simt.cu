// fp32 grouped expert GEMM on the SIMT FMA pipes (the fp32 dtype path).
//
// tcgen05 has no fp32-input kind and TF32 (10-bit mantissa) cannot hold fp32 parity, so fp32
// layers run here: one CTA per (expert, 32-row slice of a 128-row tile, 32-column tile), 256
// threads with a 2x2 register tile each (slices past the expert's rows exit at once, so the work
// follows the real row count), K staged through shared memory 32 at a time by cp.async in a ring of
// three to five slabs, so several slabs' load latencies overlap each other and the FMAs (these layers
// are small: latency, not FMA throughput, sets their time).  Every output sums its products in
// ascending k, as a plain loop would.  Each expert is
// an affine layer out = in W^T (+ b) with W stored [out, in] (hnwysp.cn/news/30485 3.2), two layers per expert
// W1 | b1 | W2 | b2 (m.nxbn.cn/news/48047 3.1), the activation applied in the epilogue
// (m.nxbn.cn 2.1: matmul and activation fused per expert).  With two slots and an fp32 output the
// down projection's epilogue also does the combine (m.nxbn.cn 3.3): g * y added onto the cleared
// output row of the row's token.
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int SBM = 32, SBN = 32, SBK = 32;
// Shared rows of 36 words: 16-byte aligned for the 16-byte copies and loads, and the 16-byte column
// reads of 8 consecutive rows (a quarter warp) land in 8 different 16-byte bank groups.
constexpr int SLD = SBK + 4;
constexpr int kSlices = kRowTile / SBM;  // row slices per 128-row tile
constexpr int TM = SBM / 16;             // rows per thread: ty * TM + i
constexpr int TN = SBN / 16;             // columns per thread: tx + 16 * j
static_assert(SBM * SBK / 4 == 256 && SBN * SBK / 4 == 256, "one 16-byte copy per thread and tile");

// 16-byte asynchronous copy global -> shared; an invalid piece is zero-filled (no bytes read)
__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemmArgs a) {
  constexpr bool kSwiGLU = EPI == kEpiSwiGLU;
  constexpr int NS = kSwiGLU ? 3 : 5;  // K slabs in flight (shared memory stays under 48 KB)
  constexpr int NB = kSwiGLU ? 2 : 1;  // weight tiles per slab (gate and up for SwiGLU)
  __shared__ __align__(16) float As[NS][SBM][SLD];
  __shared__ __align__(16) float Bs[NS][NB][SBN][SLD];
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

  // slab ks (K columns k0 = ks*SBK ...) into ring slot st, rows as stored (no transpose): thread tid
  // copies 4 consecutive k of row tid / 8 of each tile (K is a multiple of 8, so a piece is wholly
  // inside or wholly past K)
  auto load_slab = [&](int st, int k0) {
    const int r = tid >> 3, k = (tid & 7) * 4;
    const bool ink = k0 + k < a.K;
    cp_async16(&As[st][r][k], ink ? A + (size_t)(row0 + r) * a.K + k0 + k : A, ink);
    const bool in = ink && n0 + r < a.N;
    const size_t off = (size_t)(n0 + r) * a.K + k0 + k;
    cp_async16(&Bs[st][0][r][k], in ? B + off : B, in);
    if constexpr (kSwiGLU) cp_async16(&Bs[st][NB - 1][r][k], in ? B3 + off : B3, in);
  };
  const int nslab = (a.K + SBK - 1) / SBK;
#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    if (st < nslab) load_slab(st, st * SBK);
    cp_async_commit();
  }
  for (int ks = 0; ks < nslab; ++ks) {
    cp_async_wait<NS - 2>();  // this thread's copies of slab ks have landed
    __syncthreads();          // everyone's have, and every thread is done with slab ks - 1's slot
    {
      const int nx = ks + NS - 1;
      if (nx < nslab) load_slab(nx % NS, nx * SBK);
      cp_async_commit();
    }
    const int st = ks % NS;
#pragma unroll
    for (int k4 = 0; k4 < SBK; k4 += 4) {  // four k per 16-byte load, taken in ascending k
      float4 af[TM], bf[TN], bf3[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) af[i] = *reinterpret_cast<const float4*>(&As[st][ty * TM + i][k4]);
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        bf[j] = *reinterpret_cast<const float4*>(&Bs[st][0][tx + 16 * j][k4]);
        if constexpr (kSwiGLU) bf3[j] = *reinterpret_cast<const float4*>(&Bs[st][NB - 1][tx + 16 * j][k4]);
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          acc[i][j] = fmaf(af[i].x, bf[j].x, acc[i][j]);
          acc[i][j] = fmaf(af[i].y, bf[j].y, acc[i][j]);
          acc[i][j] = fmaf(af[i].z, bf[j].z, acc[i][j]);
          acc[i][j] = fmaf(af[i].w, bf[j].w, acc[i][j]);
          if constexpr (kSwiGLU) {
            acc3[i][j] = fmaf(af[i].x, bf3[j].x, acc3[i][j]);
            acc3[i][j] = fmaf(af[i].y, bf3[j].y, acc3[i][j]);
            acc3[i][j] = fmaf(af[i].z, bf3[j].z, acc3[i][j]);
            acc3[i][j] = fmaf(af[i].w, bf3[j].w, acc3[i][j]);
          }
        }
    }
  }
  cp_async_wait<0>();  // no copy in flight when the CTA leaves (the trailing groups are empty)

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = row0 + ty * TM + i;
    if (r >= seg_end) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int col = n0 + tx + 16 * j;
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
