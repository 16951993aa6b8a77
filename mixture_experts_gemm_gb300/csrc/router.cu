// Router: logits GEMM + top-2 + gates + per-chunk expert histogram, and (last CTA) the scan that
// turns the histograms into expert segment offsets.
//
// Routing follows zskr.cn/news/2272131 ("Colibri: a lightweight C MoE inference engine for edge
// devices") 3.2: routing logits, then a deterministic top-k, then per-expert counts turned into
// dispatch offsets; and hnwysp.cn/news/30485 3.1: experts returned in descending score order.
// Selection is made on the logits (softmax is monotone); ties go to the lower expert index; the
// gates are the softmax over the selected pair, g_a = 1 / (1 + exp(L_b - L_a)), g_b = 1 - g_a.
//
// The kernel is HBM-bound on reading x (2*T*E*d FLOP against T*d*sizeof(x) bytes): each warp
// streams 4 token rows with 16-byte loads while W_r sits in shared memory, so every W_r value read
// from shared memory feeds 4 tokens.  Per-chunk histograms make the dispatch deterministic: atomics
// only count finished CTAs, and every row index comes from a scan in token order.
#include "moe_internal.cuh"

namespace colibri {
namespace {

template <typename Tin>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float (&v)[4]) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <typename Tin>
__device__ __forceinline__ void load_global_vec(const Tin* p, float (&v)[Vec<Tin>::N]) {
  Vec<Tin>::load(p, v);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == kRouterThreads).  Returns the
// exclusive prefix; *total receives the block sum.
__device__ int block_exclusive_scan(int v, int* scratch /* >= 8 ints */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  int warp_prefix = 0, sum = 0;
#pragma unroll
  for (int w = 0; w < kRouterThreads / 32; ++w) {
    int s = scratch[w];
    if (w < warp) warp_prefix += s;
    sum += s;
  }
  __syncthreads();
  *total = sum;
  return warp_prefix + inc - v;
}

// Runs in the last router CTA: counts, padded offsets, M-tile prefix, and first row of each
// (chunk, expert) pair, written over the per-chunk counts.
__device__ void scan_offsets(const RouterArgs& a, int nchunks) {
  __shared__ int s_scratch[8];
  __shared__ int s_offsets[kMaxE + 1];
  const int E = a.E;
  const int per = (nchunks + kRouterThreads - 1) / kRouterThreads;
  const int c0 = threadIdx.x * per;
  const int c1 = min(c0 + per, nchunks);
  int prefix[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) {
    prefix[e] = 0;
    if (e < E) {
      int local = 0;
      for (int c = c0; c < c1; ++c) local += __ldcg(&a.hist[c * E + e]);
      int total;
      prefix[e] = block_exclusive_scan(local, s_scratch, &total);
      if (threadIdx.x == 0) a.sched->counts[e] = total;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, mt = 0;
    for (int e = 0; e < E; ++e) {
      const int c = a.sched->counts[e];
      s_offsets[e] = off;
      a.sched->offsets[e] = off;
      a.sched->mtile_start[e] = mt;
      const int tiles = (c + kRowTile - 1) / kRowTile;
      off += tiles * kRowTile;
      mt += tiles;
    }
    s_offsets[E] = off;
    a.sched->offsets[E] = off;
    a.sched->mtile_start[E] = mt;
    a.sched->ticket = 0;  // ready for the next forward
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) {
    if (e < E) {
      int run = s_offsets[e] + prefix[e];
      for (int c = c0; c < c1; ++c) {
        const int n = __ldcg(&a.hist[c * E + e]);
        a.hist[c * E + e] = run;
        run += n;
      }
    }
  }
}

template <typename Tin, int EMAX>
__global__ void __launch_bounds__(kRouterThreads) router_top2_kernel(RouterArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int VEC = Vec<Tin>::N;
  Tin* wsm = reinterpret_cast<Tin*>(smem_raw);
  __shared__ int s_idx[kRouterChunk][2];
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_t0 = blockIdx.x * kRouterChunk;
  const int t0 = chunk_t0 + warp * 4;
  const int T = a.T, d = a.d, E = a.E;
  const Tin* __restrict__ x = static_cast<const Tin*>(a.x);
  const Tin* __restrict__ w = static_cast<const Tin*>(a.w_router);

  float acc[4][EMAX];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[k][e] = 0.f;

  for (int d0 = 0; d0 < d; d0 += a.dchunk) {
    const int dc = min(a.dchunk, d - d0);
    __syncthreads();
    const int nvec = dc / VEC;
    for (int i = threadIdx.x; i < E * nvec; i += kRouterThreads) {
      const int e = i / nvec, jv = i - e * nvec;
      *reinterpret_cast<uint4*>(wsm + (size_t)e * a.dchunk + jv * VEC) =
          *reinterpret_cast<const uint4*>(w + (size_t)e * d + d0 + jv * VEC);
    }
    __syncthreads();
    for (int j = lane * VEC; j < dc; j += 32 * VEC) {
      float xv[4][VEC];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (t0 + k < T) {
          load_global_vec<Tin>(x + (size_t)(t0 + k) * d + d0 + j, xv[k]);
        } else {
#pragma unroll
          for (int v = 0; v < VEC; ++v) xv[k][v] = 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < EMAX; ++e) {
        if (e < E) {
          float wv[VEC];
          Vec<Tin>::load(wsm + (size_t)e * a.dchunk + j, wv);
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int v = 0; v < VEC; ++v) acc[k][e] = fmaf(xv[k][v], wv[v], acc[k][e]);
        }
      }
    }
  }

  // warp all-reduce: every lane ends with the full dot products
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[k][e] += __shfl_xor_sync(0xffffffffu, acc[k][e], o);

#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (lane == k) {
      const int t = t0 + k;
      float L[EMAX];
#pragma unroll
      for (int e = 0; e < EMAX; ++e) L[e] = acc[k][e] + ((a.b_router != nullptr && e < E) ? a.b_router[e] : 0.f);
      // first: highest logit, lowest index on ties (strict > keeps the earlier index)
      int ia = 0;
      float la = L[0];
#pragma unroll
      for (int e = 1; e < EMAX; ++e)
        if (e < E && L[e] > la) { la = L[e]; ia = e; }
      int ib = -1;
      float lb = 0.f;
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        if (e < E && e != ia && (ib < 0 || L[e] > lb)) { lb = L[e]; ib = e; }
      s_idx[warp * 4 + k][0] = ia;
      s_idx[warp * 4 + k][1] = ib;
      if (t < T) {
        const float ga = 1.0f / (1.0f + expf(lb - la));
        a.idx[2 * (size_t)t] = ia;
        a.idx[2 * (size_t)t + 1] = ib;
        a.gate[2 * (size_t)t] = ga;
        a.gate[2 * (size_t)t + 1] = 1.0f - ga;
      }
    }
  }
  __syncthreads();

  const int valid = min(kRouterChunk, T - chunk_t0);
  if (threadIdx.x < 2 * kRouterChunk) {
    const int tt = threadIdx.x >> 1, s = threadIdx.x & 1;
    if (tt < valid) {
      const int e = s_idx[tt][s];
      int r = 0;
      for (int u = 0; u < tt; ++u) r += (s_idx[u][0] == e) + (s_idx[u][1] == e);
      a.rank[2 * (size_t)(chunk_t0 + tt) + s] = r;
    }
  }
  if (threadIdx.x < E) {
    int c = 0;
    for (int u = 0; u < valid; ++u) c += (s_idx[u][0] == (int)threadIdx.x) + (s_idx[u][1] == (int)threadIdx.x);
    a.hist[(size_t)blockIdx.x * E + threadIdx.x] = c;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&a.sched->ticket, 1u) == gridDim.x - 1);
  __syncthreads();
  if (s_last) {
    __threadfence();
    scan_offsets(a, gridDim.x);
  }
}

template <typename Tin, int EMAX>
cudaError_t launch_router_t(const RouterArgs& a, int nchunks, cudaStream_t s) {
  const int smem = EMAX * a.dchunk * (int)sizeof(Tin);
  auto k = router_top2_kernel<Tin, EMAX>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  k<<<nchunks, kRouterThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int router_smem_bytes(int dtype, int E, int dchunk) {
  const int emax = E <= 4 ? 4 : (E <= 8 ? 8 : 16);
  return emax * dchunk * (dtype == 0 ? 4 : 2);
}

cudaError_t launch_router(int dtype, const RouterArgs& a, int nchunks, cudaStream_t s) {
  if (dtype == 0) {
    if (a.E <= 4) return launch_router_t<float, 4>(a, nchunks, s);
    if (a.E <= 8) return launch_router_t<float, 8>(a, nchunks, s);
    return launch_router_t<float, 16>(a, nchunks, s);
  }
  if (a.E <= 4) return launch_router_t<__nv_bfloat16, 4>(a, nchunks, s);
  if (a.E <= 8) return launch_router_t<__nv_bfloat16, 8>(a, nchunks, s);
  return launch_router_t<__nv_bfloat16, 16>(a, nchunks, s);
}

}  // namespace colibri
