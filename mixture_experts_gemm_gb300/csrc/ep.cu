// Expert parallelism: the layer's experts split over ep_size GPUs, one process per GPU.
//
// A token's rows go to the GPUs that own its experts and its expert outputs come back to it for the
// combine.  The articles run one device (no collectives); the split follows the Dispatch /
// Compute stages of zskr.cn/news/2272131 ("Colibri: a lightweight C MoE inference engine for edge
// devices") 2.1, with the exchange between the two stages:
//   source rank:  router (all E experts) -> ep_pack: x rows grouped by expert, ascending token
//                 inside each expert, unpadded ("send rows"), so rank q's rows are one contiguous
//                 block (experts q*El .. q*El+El-1)
//   exchange:     all-to-all of the per-expert counts, then of the rows (caller's communicator)
//   expert rank:  ep_regroup: received rows (source-major: source p, local expert j) into 128-row
//                 padded expert segments (expert-major: j, then p) and the local schedule ->
//                 grouped up / down GEMMs; the CTA-pair down GEMM writes each fp32 row straight to its
//                 receive position (a row map the regroup fills), other kernels write Y and
//                 ep_unregroup copies it back to receive order
//   exchange:     all-to-all of the output rows back to their sources
//   source rank:  combine over the returned rows (the forward's combine kernel).
// Every copy is a plain HBM-bound row copy: one warp per row, 16-byte vectors.
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int kEpThreads = 256;

// Send rows: row_of[t, s] (rank inside the router chunk) -> position in the send buffer; the token
// row copied there.  Position = unpadded start of the expert + rank of t among the expert's tokens
// (= first padded row of (chunk, expert) + rank in chunk - padded start of the expert).
template <int ESIZE>
__global__ void __launch_bounds__(kEpThreads) ep_pack_kernel(EpPackArgs a, int wpt) {
  __shared__ int s_raw[kMaxE], s_pad[kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (kEpThreads / 32) + warp;
  const int t = gw / wpt, part = gw - t * wpt;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < a.E; ++e) {
      s_raw[e] = acc;
      s_pad[e] = a.sched->offsets[e];
      acc += a.sched->counts[e];
    }
  }
  if (blockIdx.x == 0 && threadIdx.x < a.E) a.send_counts[threadIdx.x] = a.sched->counts[threadIdx.x];
  __syncthreads();
  const bool valid = t < a.T;
  const int k = a.k;
  const int n_rows = a.T * k;
  int r[kMaxTopK];
  bool ok = valid;
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    r[s] = 0;
    if (valid && s < k) {
      const int e = a.idx[(size_t)k * t + s];
      r[s] = a.chunk_base[(size_t)(t / kRouterChunk) * a.E + e] + a.row_of[(size_t)k * t + s] - s_pad[e] + s_raw[e];
      ok = ok && r[s] >= 0 && r[s] < n_rows;
    }
  }
  __syncthreads();  // every warp of the token has read the ranks before they are overwritten
  if (!valid) return;
  if (lane == 0 && part == 0) {
    if (ok) {
      for (int s = 0; s < k; ++s) a.row_of[(size_t)k * t + s] = r[s];
    } else {
      atomicOr(a.status, kStatusBadRow);
    }
  }
  if (!ok) return;
  const size_t row_bytes = (size_t)a.d * ESIZE;
  const int nvec = (int)(row_bytes / 16);
  const int v0 = (nvec * part) / wpt, v1 = (nvec * (part + 1)) / wpt;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.x) + (size_t)t * row_bytes);
  char* dst = static_cast<char*>(a.send);
  for (int i = v0 + lane; i < v1; i += 32) {
    const uint4 q = __ldg(src + i);
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s)
      if (s < k) reinterpret_cast<uint4*>(dst + (size_t)r[s] * row_bytes)[i] = q;
  }
}

// Segment of received row i (receive order): the (source, local expert) block holding it.
__device__ __forceinline__ int ep_segment(const EpPlan& p, int i) {
  int g = 0;
  while (g + 1 < p.n_seg && i >= p.src[g + 1]) ++g;
  return g;
}

// Received rows into the padded expert segments of Xp; block 0 also writes the local schedule.
__global__ void __launch_bounds__(kEpThreads) ep_regroup_kernel(EpRegroupArgs a) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    const int E = a.plan.El;
    if (threadIdx.x < E) a.sched->counts[threadIdx.x] = a.plan.counts[threadIdx.x];
    if (threadIdx.x <= E) {
      a.sched->offsets[threadIdx.x] = a.plan.offsets[threadIdx.x];
      a.sched->mtile_start[threadIdx.x] = a.plan.mstart[threadIdx.x];
    }
    if (threadIdx.x == 0) reset_gemm_counters(a.sched);
  }
  const int nvec = a.row_bytes / 16;
  const int warps = gridDim.x * (kEpThreads / 32);
  for (int i = blockIdx.x * (kEpThreads / 32) + (threadIdx.x >> 5); i < a.R; i += warps) {
    const int g = ep_segment(a.plan, i);
    const int dst = a.plan.dst[g] + (i - a.plan.src[g]);
    if (a.recv_of_row != nullptr && (threadIdx.x & 31) == 0) a.recv_of_row[dst] = i;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(a.recv) + (size_t)i * a.row_bytes);
    uint4* out = reinterpret_cast<uint4*>(static_cast<char*>(a.xp) + (size_t)dst * a.row_bytes);
    for (int v = threadIdx.x & 31; v < nvec; v += 32) out[v] = __ldg(src + v);
  }
}

// Expert outputs (fp32 Y rows of the padded layout) back to receive order.
__global__ void __launch_bounds__(kEpThreads) ep_unregroup_kernel(EpUnregroupArgs a) {
  pdl_trigger();
  pdl_wait();
  const int nvec = a.d / 4;
  const int warps = gridDim.x * (kEpThreads / 32);
  for (int i = blockIdx.x * (kEpThreads / 32) + (threadIdx.x >> 5); i < a.R; i += warps) {
    const int g = ep_segment(a.plan, i);
    const int row = a.plan.dst[g] + (i - a.plan.src[g]);
    const float4* src = reinterpret_cast<const float4*>(a.y + (size_t)row * a.d);
    float4* out = reinterpret_cast<float4*>(a.y_out + (size_t)i * a.d);
    for (int v = threadIdx.x & 31; v < nvec; v += 32) __stcs(out + v, __ldcs(src + v));
  }
}

int copy_grid(int rows, int num_sms) {
  const int per = kEpThreads / 32;
  const int need = (rows + per - 1) / per;
  return need < num_sms * 8 ? need : num_sms * 8;
}

}  // namespace

cudaError_t launch_ep_pack(int dtype, const EpPackArgs& a, cudaStream_t s) {
  const int per = kEpThreads / 32;
  const int wpt = a.T >= 1024 ? 1 : (a.T >= 256 ? 2 : (a.T >= 64 ? 4 : 8));
  const int grid = (a.T * wpt + per - 1) / per;
  if (dtype == 0) return pdl_launch(ep_pack_kernel<4>, dim3(grid), dim3(kEpThreads), 0, s, a, wpt);
  return pdl_launch(ep_pack_kernel<2>, dim3(grid), dim3(kEpThreads), 0, s, a, wpt);
}

cudaError_t launch_ep_regroup(const EpRegroupArgs& a, int num_sms, cudaStream_t s) {
  const int grid = a.R > 0 ? copy_grid(a.R, num_sms) : 1;
  return pdl_launch(ep_regroup_kernel, dim3(grid), dim3(kEpThreads), 0, s, a);
}

cudaError_t launch_ep_unregroup(const EpUnregroupArgs& a, int num_sms, cudaStream_t s) {
  return pdl_launch(ep_unregroup_kernel, dim3(copy_grid(a.R, num_sms)), dim3(kEpThreads), 0, s, a);
}

}  // namespace colibri
