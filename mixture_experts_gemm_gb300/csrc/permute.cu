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
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherArgs a, int wpt) {
  // wpt warps share one token row (small batches spread a row over several warps)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kGatherThreads / 32) + warp;
  const int t = gw / wpt, part = gw - t * wpt;
  pdl_wait();
  pdl_trigger();  // after the wait: the next kernel may then read what the router wrote before waiting
  const bool valid = t < a.T;
  const int chunk = t / kRouterChunk;
  const int S = a.S;
  int r[kMaxSlots];
  bool ok = valid;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    r[s] = 0;
    if (valid && s < S) {
      const int e = a.idx[(size_t)S * t + s];
      r[s] = a.chunk_base[(size_t)chunk * a.E + e] + a.row_of[(size_t)S * t + s];
      ok = ok && r[s] >= 0 && r[s] < a.rows_alloc;
    }
  }
  // the wpt warps of a token (all in this CTA) have read its in-chunk ranks before the first warp
  // overwrites them with rows below
  __syncthreads();
  if (!valid) return;
  if (lane == 0 && part == 0) {
    if (ok) {
      for (int s = 0; s < S; ++s) {
        a.row_of[(size_t)S * t + s] = r[s];
        a.token_of_row[r[s]] = t;
        if (a.gate_of_row) a.gate_of_row[r[s]] = a.gate[(size_t)S * t + s];
      }
    } else {
      atomicOr(&a.sched->status, kStatusBadRow);
    }
  }
  if (!ok) return;

  const size_t row_bytes = (size_t)a.d * ESIZE;
  const int nvec = (int)(row_bytes / 16);
  const int v0 = (nvec * part) / wpt, v1 = (nvec * (part + 1)) / wpt;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)t * row_bytes);
  char* xp = static_cast<char*>(a.xp);
  if (S == 2) {
    uint4* d0 = reinterpret_cast<uint4*>(xp + (size_t)r[0] * row_bytes);
    uint4* d1 = reinterpret_cast<uint4*>(xp + (size_t)r[1] * row_bytes);
    int i = v0 + lane;
    for (; i + 96 < v1; i += 128) {
      uint4 q0 = __ldg(src + i), q1 = __ldg(src + i + 32), q2 = __ldg(src + i + 64), q3 = __ldg(src + i + 96);
      d0[i] = q0; d0[i + 32] = q1; d0[i + 64] = q2; d0[i + 96] = q3;
      d1[i] = q0; d1[i + 32] = q1; d1[i + 64] = q2; d1[i + 96] = q3;
    }
    for (; i < v1; i += 32) {
      uint4 q = __ldg(src + i);
      d0[i] = q;
      d1[i] = q;
    }
  } else {
    for (int i = v0 + lane; i < v1; i += 32) {
      const uint4 q = __ldg(src + i);
#pragma unroll
      for (int s = 0; s < kMaxSlots; ++s)
        if (s < S) reinterpret_cast<uint4*>(xp + (size_t)r[s] * row_bytes)[i] = q;
    }
  }
}

// Bookkeeping only, for the path whose up GEMM gathers its A rows from x itself: one thread per
// token, same rows as gather_kernel.
__global__ void __launch_bounds__(kGatherThreads) dispatch_rows_kernel(GatherArgs a) {
  const int t = blockIdx.x * kGatherThreads + threadIdx.x;
  pdl_wait();
  pdl_trigger();  // after the wait: the next kernel may then read what the router wrote before waiting
  if (t >= a.T) return;
  const int chunk = t / kRouterChunk;
  const int S = a.S;
  int r[kMaxSlots];
  bool ok = true;
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s) {
    r[s] = 0;
    if (s < S) {
      const int e = a.idx[(size_t)S * t + s];
      r[s] = a.chunk_base[(size_t)chunk * a.E + e] + a.row_of[(size_t)S * t + s];
      ok = ok && r[s] >= 0 && r[s] < a.rows_alloc;
    }
  }
  if (!ok) {
    atomicOr(&a.sched->status, kStatusBadRow);
    return;
  }
#pragma unroll
  for (int s = 0; s < kMaxSlots; ++s)
    if (s < S) {
      a.row_of[(size_t)S * t + s] = r[s];
      a.token_of_row[r[s]] = t;
      if (a.gate_of_row) a.gate_of_row[r[s]] = a.gate[(size_t)S * t + s];
    }
}

}  // namespace

cudaError_t launch_gather(int dtype, const GatherArgs& a, cudaStream_t s) {
  if (a.xp == nullptr)
    return pdl_launch(dispatch_rows_kernel, dim3((a.T + kGatherThreads - 1) / kGatherThreads), dim3(kGatherThreads),
                      0, s, a);
  const int per = kGatherThreads / 32;
  const int wpt = a.T >= 1024 ? 1 : (a.T >= 256 ? 2 : (a.T >= 64 ? 4 : 8));
  const int grid = (a.T * wpt + per - 1) / per;
  if (dtype == 0) return pdl_launch(gather_kernel<4>, dim3(grid), dim3(kGatherThreads), 0, s, a, wpt);
  return pdl_launch(gather_kernel<2>, dim3(grid), dim3(kGatherThreads), 0, s, a, wpt);
}

}  // namespace colibri
