// Dispatch gather: token rows copied into expert-contiguous rows (Xp), plus the row bookkeeping.
//
// zskr.cn/news/2272131 ("Colibri: a lightweight C MoE inference engine for edge devices") 2.1:
// the Dispatch stage groups tokens by expert so the Compute stage can run one GEMM per expert;
// 3.2: "sort tokens by expert index" from the per-expert counts.  Rows inside one expert's
// segment follow ascending token index (a counting sort): row = first row of (chunk, expert) from
// the router's scan + the token's rank inside its chunk.
//
// HBM-bound copy: each token row is read once and written twice (its two experts).  One warp per
// token, 16-byte vector loads and stores, four loads in flight per lane.
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int kGatherThreads = 256;

template <int ESIZE>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kGatherThreads / 32) + warp;
  if (t >= a.T) return;
  const int chunk = t / kRouterChunk;
  int r[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int e = a.idx[2 * (size_t)t + s];
    r[s] = a.chunk_base[(size_t)chunk * a.E + e] + a.row_of[2 * (size_t)t + s];
  }
  const bool ok = r[0] >= 0 && r[0] < a.rows_alloc && r[1] >= 0 && r[1] < a.rows_alloc;
  __syncwarp();
  if (lane == 0) {
    if (ok) {
      a.row_of[2 * (size_t)t] = r[0];
      a.row_of[2 * (size_t)t + 1] = r[1];
      a.token_of_row[r[0]] = t;
      a.token_of_row[r[1]] = t;
    } else {
      atomicOr(&a.sched->status, kStatusBadRow);
    }
  }
  if (!ok) return;
  const size_t row_bytes = (size_t)a.d * ESIZE;
  const int nvec = (int)(row_bytes / 16);
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)t * row_bytes);
  uint4* d0 = reinterpret_cast<uint4*>(static_cast<char*>(a.xp) + (size_t)r[0] * row_bytes);
  uint4* d1 = reinterpret_cast<uint4*>(static_cast<char*>(a.xp) + (size_t)r[1] * row_bytes);
  int i = lane;
  for (; i + 96 < nvec; i += 128) {
    uint4 v0 = __ldg(src + i), v1 = __ldg(src + i + 32), v2 = __ldg(src + i + 64), v3 = __ldg(src + i + 96);
    d0[i] = v0; d0[i + 32] = v1; d0[i + 64] = v2; d0[i + 96] = v3;
    d1[i] = v0; d1[i + 32] = v1; d1[i + 64] = v2; d1[i + 96] = v3;
  }
  for (; i < nvec; i += 32) {
    uint4 v = __ldg(src + i);
    d0[i] = v;
    d1[i] = v;
  }
}

}  // namespace

cudaError_t launch_gather(int dtype, const GatherArgs& a, cudaStream_t s) {
  const int per = kGatherThreads / 32;
  const int grid = (a.T + per - 1) / per;
  if (dtype == 0)
    gather_kernel<4><<<grid, kGatherThreads, 0, s>>>(a);
  else
    gather_kernel<2><<<grid, kGatherThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace colibri
