// colibri_moe_route_noalloc: the routing stage (router kernel + row bookkeeping) for callers that
// cannot allocate device memory.  Its scratch -- the per-chunk expert histograms and the routing
// summary the router's last CTA writes -- lives in one file-scope __device__ array instead of a
// context's workspace, so the call needs no context and never allocates.
//
// The array is a fixed part of the library's device image: every GPU that loads the library holds
// it (kNoAllocScratchBytes) until the process exits.  Host code may not use the array's name as a
// device address; the address comes from cudaGetSymbolAddress, once per device, at first use.
#include <mutex>

#include "colibri_moe.h"
#include "moe_internal.cuh"

namespace colibri {
namespace {

constexpr int kNoAllocMaxTokens = 65536;
constexpr int kNoAllocMaxChunks = kNoAllocMaxTokens / kRouterChunk;           // 2048
constexpr size_t kSchedBytes = (sizeof(Sched) + 255) / 256 * 256;
constexpr size_t kNoAllocScratchBytes = kSchedBytes + size_t(kNoAllocMaxChunks) * kMaxE * sizeof(int32_t);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_route_scratch on `device` (the current device), looked up once.
cudaError_t scratch_address(int device, void** out) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    for (int dtype = 0; dtype < 2; ++dtype)
      for (int E : {4, 8, 16}) {
        e = prepare_router(dtype, E);
        if (e != cudaSuccess) return e;
      }
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

// row_of[t, s] = first row of (chunk, expert) + rank inside the chunk; counts and offsets copied out.
__global__ void route_rows_kernel(const int32_t* __restrict__ idx, int32_t* __restrict__ row_of,
                                  const int32_t* __restrict__ chunk_base, const Sched* __restrict__ sched, int T,
                                  int E, int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 2 * T) {
    const int t = i >> 1;
    row_of[i] += chunk_base[(t / kRouterChunk) * E + idx[i]];
  }
  if (blockIdx.x == 0 && threadIdx.x <= E) {
    if (threadIdx.x < E) counts[threadIdx.x] = sched->counts[threadIdx.x];
    offsets[threadIdx.x] = sched->offsets[threadIdx.x];
  }
}

bool on_device(const void* p, int device) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeManaged || (at.type == cudaMemoryTypeDevice && at.device == device);
}

}  // namespace
}  // namespace colibri

using namespace colibri;

extern "C" int colibri_moe_route_noalloc(const void* x, const void* w_router, const float* b_router, int32_t T,
                                         int32_t d_model, int32_t num_experts, int32_t dtype, int32_t* idx,
                                         float* gate, int32_t* counts, int32_t* offsets, int32_t* row_of,
                                         void* stream) {
  if (T < 0 || T > kNoAllocMaxTokens) return COLIBRI_ERR_INVALID_ARG;
  if (num_experts < 2 || num_experts > kMaxRouted || d_model <= 0) return COLIBRI_ERR_INVALID_ARG;
  if (dtype != COLIBRI_DTYPE_F32 && dtype != COLIBRI_DTYPE_BF16) return COLIBRI_ERR_INVALID_ARG;
  if (d_model % 8) return COLIBRI_ERR_UNSUPPORTED;
  if (!counts || !offsets || (T > 0 && (!x || !w_router || !idx || !gate || !row_of))) return COLIBRI_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  const void* dev_ptrs[] = {x, w_router, b_router, idx, gate, counts, offsets, row_of};
  for (const void* p : dev_ptrs)
    if (p && !on_device(p, device)) return COLIBRI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15) return COLIBRI_ERR_INVALID_ARG;

  void* scratch = nullptr;
  if (scratch_address(device, &scratch) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Sched* sched = static_cast<Sched*>(scratch);
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + kSchedBytes);
  const int E = num_experts;
  // the router's CTA ticket and the status word must start at zero; histograms are fully rewritten
  if (cudaMemsetAsync(sched, 0, sizeof(Sched), s) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, E * sizeof(int32_t), s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s) != cudaSuccess) {
      cudaGetLastError();
      return COLIBRI_ERR_CUDA;
    }
    return COLIBRI_OK;
  }
  const int esize = dtype == COLIBRI_DTYPE_F32 ? 4 : 2;
  const int vec_span = 32 * (16 / esize);
  const int emax = E <= 4 ? 4 : (E <= 8 ? 8 : 16);
  int dchunk = kRouterMaxSmem / (emax * esize) / vec_span * vec_span;
  if (d_model < dchunk) dchunk = d_model;
  const int nchunks = (T + kRouterChunk - 1) / kRouterChunk;
  RouterArgs ra{x, w_router, b_router, T, d_model, E, dchunk, idx, gate, row_of, hist, sched, 2, 0, 0, 2, E};
  if (launch_router(dtype, ra, nchunks, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  const int threads = 256;
  route_rows_kernel<<<(2 * T + threads - 1) / threads, threads, 0, s>>>(idx, row_of, hist, sched, T, E, counts,
                                                                          offsets);
  if (cudaGetLastError() != cudaSuccess) return COLIBRI_ERR_CUDA;
  return COLIBRI_OK;
}
