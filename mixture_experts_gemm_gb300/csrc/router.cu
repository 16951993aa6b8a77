// Router: logits GEMM + top-2 + gates + per-chunk expert histogram, and (last CTA) the scan that
// turns the histograms into expert segment offsets.
//
// Routing follows zskr.cn/news/2272131 ("Colibri: a lightweight C MoE inference engine for edge
// devices") 3.2: routing logits, then a deterministic top-k, then per-expert counts turned into
// dispatch offsets; and hnwysp.cn/news/30485 3.1: experts returned in descending score order.
// Selection is made on the logits (softmax is monotone); ties go to the lower expert index; the
// gates are the softmax over the selected pair, g_a = 1 / (1 + exp(L_b - L_a)), g_b = 1 - g_a.
//
// The work is bound by reading x (2*T*E*d FLOP against T*d*sizeof(x) bytes).  One CTA per 32-token
// chunk; four kernels share the top-k, histogram and scan code below:
//   router_top2_kernel      fp32 (and bf16 with d not a multiple of 32): FMA dot products, W_r
//                           staged in shared memory, each warp streaming 4 token rows;
//   router_top2_mma_kernel  bf16: mma.sync logits with fragments loaded straight from x;
//   router_split_kernel     bf16, 9..1024 tokens: d split over 8 CTAs per chunk;
//   router_tma_kernel       bf16, >= 1024 tokens: x staged through shared memory by TMA.
// Per-chunk histograms make the dispatch deterministic: atomics only count finished CTAs, and every
// row index comes from a scan in token order.
#include <utility>

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
  __device__ static void from_raw(const uint4& q, float (&v)[4]) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void from_raw(const uint4& q, float (&v)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    from_raw(*reinterpret_cast<const uint4*>(p), v);
  }
};

// Runs in the last router CTA: counts, padded offsets, M-tile prefix, and the first row of every
// (chunk, expert) pair, written over the per-chunk counts.  Thread t owns a contiguous range of
// chunks and reads every expert's count of a chunk at once (independent loads, one L2 round trip
// per chunk of its range); a block-wide exclusive scan over the threads, per expert, then gives every
// chunk's place in chunk order.  Thread 0 turns the expert totals into padded segment offsets.
__device__ void scan_offsets(const RouterArgs& a, int nchunks) {
  constexpr int NTH = kRouterThreads, NW = NTH / 32;
  __shared__ int s_wsum[NW][kMaxE];  // per-warp totals, then their exclusive prefix over warps
  __shared__ int s_tot[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  const int E = a.Ex;  // scheduled experts: routed (+ shared)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nchunks + NTH - 1) / NTH;
  const int c0 = min(tid * per, nchunks), c1 = min(c0 + per, nchunks);
  int sum[kMaxE], first[kMaxE];  // first: the counts of chunk c0, kept for the second pass
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) sum[e] = first[e] = 0;
  for (int c = c0; c < c1; ++c) {
    int v[kMaxE];
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) v[e] = e < E ? __ldcg(&a.hist[(size_t)c * E + e]) : 0;
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) sum[e] += v[e];
    if (c == c0) {
#pragma unroll
      for (int e = 0; e < kMaxE; ++e) first[e] = v[e];
    }
  }
  int excl[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) {
    int inc = sum[e];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += n;
    }
    excl[e] = inc - sum[e];
    if (lane == 31) s_wsum[warp][e] = inc;
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
    for (int w = 0; w < NW; ++w) {
      const int t = s_wsum[w][tid];
      s_wsum[w][tid] = run;
      run += t;
    }
    s_tot[tid] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, mt = 0;
    for (int e = 0; e < E; ++e) {
      const int tot = s_tot[e];
      s_off[e] = off;
      a.sched->counts[e] = tot;
      a.sched->offsets[e] = off;
      a.sched->mtile_start[e] = mt;
      const int tiles = (tot + kRowTile - 1) / kRowTile;
      off += tiles * kRowTile;
      mt += tiles;
    }
    s_off[E] = off;
    a.sched->offsets[E] = off;
    a.sched->mtile_start[E] = mt;
    a.sched->ticket = 0;  // ready for the next forward
    a.sched->grid_sync = 0;
    reset_gemm_counters(a.sched);
    for (int i = 0; i < a.n_tile_done; ++i) a.tile_done[i] = 0;  // (normally already 0: self-resetting)
  }
  __syncthreads();
  int run[kMaxE];
#pragma unroll
  for (int e = 0; e < kMaxE; ++e) run[e] = e < E ? s_off[e] + s_wsum[warp][e] + excl[e] : 0;
  for (int c = c0; c < c1; ++c) {
    int v[kMaxE];
#pragma unroll
    for (int e = 0; e < kMaxE; ++e) v[e] = c == c0 ? first[e] : (e < E ? __ldcg(&a.hist[(size_t)c * E + e]) : 0);
#pragma unroll
    for (int e = 0; e < kMaxE; ++e)
      if (e < E) {
        a.hist[(size_t)c * E + e] = run[e];
        run[e] += v[e];
      }
  }
}

// After the chunk's routing is in s_idx (a __syncthreads() ago): in-chunk ranks, the chunk's expert
// histogram, and -- in the CTA that finishes last -- the scan of all histograms.  S slots per token
// (k routed experts, then the shared expert when present); a token names each expert at most once.
// With the dispatch fused (a.xp set) it stops after the histogram (the ranks also go to s_rank, when
// given): fused_dispatch takes over.
__device__ void finish_chunk(const RouterArgs& a, const int (*s_idx)[kMaxSlots], int valid, int chunk_t0,
                             int chunk = blockIdx.x, int nchunks = gridDim.x, int* s_rank = nullptr) {
  __shared__ int s_last;
  // The chunk's (token, slot) entries in token-major order, one per thread of the first warps.  An
  // entry's rank is the number of earlier entries naming its expert (no token names an expert twice,
  // so these are the earlier tokens' rows of that expert): the warp's equal-expert lanes below it,
  // plus the earlier warps' counts of that expert.
  __shared__ int s_wcnt[kMaxSlots][kMaxE];  // entries of warp w naming expert e
  const int Ex = a.Ex, S = a.S;
  const int n = valid * S, nw = (n + 31) >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int e_ent = -1;
  unsigned same = 0;
  if (warp < nw) {
    const int i = threadIdx.x;
    e_ent = i < n ? s_idx[i / S][i - (i / S) * S] : -1;
    same = __match_any_sync(0xffffffffu, e_ent);
    if (lane < Ex) s_wcnt[warp][lane] = 0;
    __syncwarp();
    if (e_ent >= 0 && (same & ((1u << lane) - 1u)) == 0) s_wcnt[warp][e_ent] = __popc(same);
  }
  __syncthreads();
  if (e_ent >= 0) {
    int r = __popc(same & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w) r += s_wcnt[w][e_ent];
    a.rank[(size_t)S * chunk_t0 + threadIdx.x] = r;
    if (s_rank) s_rank[threadIdx.x] = r;
  }
  __shared__ int s_cnt[kMaxE];
  if (threadIdx.x < Ex) {
    int c = 0;
    for (int w = 0; w < nw; ++w) c += s_wcnt[w][threadIdx.x];
    if (nchunks > 1 || a.xp)
      a.hist[(size_t)chunk * Ex + threadIdx.x] = c;
    else
      s_cnt[threadIdx.x] = c;
  }
  if (a.xp) return;  // fused dispatch: the grid barrier and the rows follow
  if (nchunks == 1) {
    // one chunk (T <= 32, decode-sized batches): no other CTA to wait for, so the summary comes
    // straight from this CTA's counts; the chunk's first row of each expert is the expert's offset
    __syncthreads();
    if (threadIdx.x == 0) {
      int off = 0, mt = 0;
      for (int e = 0; e < Ex; ++e) {
        const int tot = s_cnt[e];
        a.sched->counts[e] = tot;
        a.sched->offsets[e] = off;
        a.sched->mtile_start[e] = mt;
        a.hist[e] = off;
        const int tiles = (tot + kRowTile - 1) / kRowTile;
        off += tiles * kRowTile;
        mt += tiles;
      }
      a.sched->offsets[Ex] = off;
      a.sched->mtile_start[Ex] = mt;
      a.sched->ticket = 0;
      a.sched->grid_sync = 0;
      reset_gemm_counters(a.sched);
      for (int i = 0; i < a.n_tile_done; ++i) a.tile_done[i] = 0;
    }
    return;
  }
  // The ticket: an acquire-release add by thread 0 after the block barrier.  Its release covers the
  // whole CTA's rank and count stores (ordered before it by the barrier; release is cumulative) and,
  // in the CTA that takes the last ticket, its acquire orders every other CTA's counts before the
  // scan's loads (the barrier after it carries that to the other threads).
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned before;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(&a.sched->ticket) : "memory");
    s_last = before == static_cast<unsigned>(nchunks) - 1u;
  }
  __syncthreads();
  if (s_last) scan_offsets(a, nchunks);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t router_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Fused dispatch, after finish_chunk has stored this chunk's histogram (and, in the CTA that
// completed the chunk, its ranks).  A grid barrier (every CTA of the cooperative launch arrives
// once, a gpu-scope release; the spin an acquire, bounded), then every CTA computes its chunk's
// first row of each expert from all chunks' counts -- the prefix over the chunks before it plus the
// 128-row padded start of the expert, the same scan the last-CTA path does, in chunk order -- and
// copies columns [col0, col1) of its tokens' rows of x into Xp (the row of token t, slot s =
// first row of (chunk, e) + rank).  The `writer` CTA of a chunk also writes row_of, token_of_row and
// gate_of_row; CTA 0 writes the routing summary.  s_rank / s_idx: the chunk's ranks and experts in
// shared memory, or nullptr to read them from global memory (the other CTAs of a split chunk).
template <int ESIZE>
__device__ void fused_dispatch(const RouterArgs& a, int chunk, int nchunks, int chunk_t0, int valid,
                               const int* s_rank, const int (*s_idx)[kMaxSlots], int col0, int col1, bool writer) {
  __shared__ int s_before[kMaxE], s_total[kMaxE], s_off[kMaxE + 1];
  __shared__ int s_row[kRouterChunk * kMaxSlots];
  __shared__ int s_go;
  const int Ex = a.Ex, S = a.S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.route_sync) : "memory");
    const uint32_t target = gridDim.x;
    int go = 1;
    if (ld_acquire_u32(a.route_sync) < target) {
      const uint64_t t0 = router_now_ns();
      while (ld_acquire_u32(a.route_sync) < target) {
        if (router_now_ns() - t0 > a.timeout_ns) {
          atomicOr(&a.sched->status, kStatusTimeoutRouteSync);
          go = 0;
          break;
        }
      }
    }
    s_go = go;
  }
  __syncthreads();
  if (!s_go) return;
  // per expert: rows of all chunks, and of the chunks before this one (one warp per expert)
  for (int e = warp; e < Ex; e += kRouterThreads / 32) {
    int tot = 0, bef = 0;
    for (int c = lane; c < nchunks; c += 32) {
      const int v = __ldcg(&a.hist[(size_t)c * Ex + e]);
      tot += v;
      bef += c < chunk ? v : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      bef += __shfl_xor_sync(0xffffffffu, bef, o);
    }
    if (lane == 0) {
      s_total[e] = tot;
      s_before[e] = bef;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, mt = 0;
    const bool summary = blockIdx.x == 0;
    for (int e = 0; e < Ex; ++e) {
      s_off[e] = off;
      const int tiles = (s_total[e] + kRowTile - 1) / kRowTile;
      if (summary) {
        a.sched->counts[e] = s_total[e];
        a.sched->offsets[e] = off;
        a.sched->mtile_start[e] = mt;
      }
      off += tiles * kRowTile;
      mt += tiles;
    }
    s_off[Ex] = off;
    if (summary) {
      a.sched->offsets[Ex] = off;
      a.sched->mtile_start[Ex] = mt;
      a.sched->ticket = 0;
      a.sched->grid_sync = 0;
      reset_gemm_counters(a.sched);
      for (int i = 0; i < a.n_tile_done; ++i) a.tile_done[i] = 0;
    }
  }
  __syncthreads();
  // rows of the chunk's (token, slot) entries
  bool bad = false;
  for (int i = threadIdx.x; i < valid * S; i += kRouterThreads) {
    const int t = i / S, sl = i - t * S;
    const size_t gi = (size_t)S * chunk_t0 + i;
    const int e = s_idx ? s_idx[t][sl] : __ldcg(&a.idx[gi]);
    const int r = s_rank ? s_rank[i] : __ldcg(&a.rank[gi]);
    const int row = s_off[e] + s_before[e] + r;
    const bool ok = e >= 0 && e < Ex && row >= 0 && row < a.rows_alloc;
    bad |= !ok;
    s_row[i] = ok ? row : -1;
    if (writer && ok) {
      a.row_of[gi] = row;
      a.token_of_row[row] = chunk_t0 + t;
      if (a.gate_of_row) a.gate_of_row[row] = a.gate[gi];
    }
  }
  if (bad) atomicOr(&a.sched->status, kStatusBadRow);
  __syncthreads();
  // copy: 16-byte vectors of columns [col0, col1) of every valid token row to its S rows of Xp
  const int vpr = (col1 - col0) * ESIZE / 16;  // vectors per row
  const size_t row_bytes = (size_t)a.d * ESIZE;
  const char* xb = static_cast<const char*>(a.x) + (size_t)col0 * ESIZE;
  char* pb = static_cast<char*>(a.xp) + (size_t)col0 * ESIZE;
  for (int i = threadIdx.x; i < valid * vpr; i += kRouterThreads) {
    const int t = i / vpr, v = i - t * vpr;
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(xb + (size_t)(chunk_t0 + t) * row_bytes) + v);
#pragma unroll
    for (int sl = 0; sl < kMaxSlots; ++sl)
      if (sl < S) {
        const int row = s_row[t * S + sl];
        if (row >= 0) reinterpret_cast<uint4*>(pb + (size_t)row * row_bytes)[v] = q;
      }
  }
}

// Top-k of one token's logits (strict > keeps the lower index on ties) and its gates:
// softmax over the selected experts (k = 2: g_a = 1 / (1 + e^{L_b - L_a}), g_b = 1 - g_a), or the
// full softmax over all experts at the selected ones (gate_mode 1).  The shared expert, when
// present, takes slot k with gate 1.
template <int EMAX>
__device__ __forceinline__ void topk_store(const RouterArgs& a, const float (&L)[EMAX], int t, int* sidx) {
  const int E = a.E, k = a.k;
  int sel[kMaxTopK];
  float ls[kMaxTopK];
  uint32_t used = 0;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    int best = -1;
    float lbest = 0.f;
    if (j < k) {
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        if (e < E && !((used >> e) & 1u) && (best < 0 || L[e] > lbest)) { lbest = L[e]; best = e; }
      used |= 1u << best;
    }
    sel[j] = best;
    ls[j] = lbest;
  }
  float g[kMaxTopK];
  if (a.gate_mode == 0 && k == 2) {
    g[0] = 1.0f / (1.0f + expf(ls[1] - ls[0]));
    g[1] = 1.0f - g[0];
  } else {
    float den = 0.f;
    if (a.gate_mode == 0) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) den += expf(ls[j] - ls[0]);
    } else {
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        if (e < E) den += expf(L[e] - ls[0]);
    }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) g[j] = j < k ? expf(ls[j] - ls[0]) / den : 0.f;
  }
  const int S = a.S;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) sidx[j] = sel[j];
  if (a.shared) sidx[k] = E;
  if (t < a.T) {
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        a.idx[(size_t)S * t + j] = sel[j];
        a.gate[(size_t)S * t + j] = g[j];
      }
    if (a.shared) {
      a.idx[(size_t)S * t + k] = E;
      a.gate[(size_t)S * t + k] = 1.0f;
    }
  }
}

// The warps' partial logit tiles (warp w holds half w % H of the chunk's rows over hidden slice
// w / H) summed in slice order, plus the router bias, for the first nrows rows: every thread takes
// some (row, expert) sums, then a __syncthreads().
template <int EMAX>
__device__ __forceinline__ void sum_slices(const RouterArgs& a, const float (*s_part)[16][EMAX],
                                           float (*s_logit)[EMAX], int H, int S, int nrows) {
  for (int i = threadIdx.x; i < nrows * EMAX; i += blockDim.x) {
    const int r = i / EMAX, e = i - r * EMAX, hh = r >> 4, rr = r & 15;
    float v = s_part[hh][rr][e];
    for (int w = 1; w < S; ++w) v += s_part[hh + w * H][rr][e];
    s_logit[r][e] = v + ((a.b_router != nullptr && e < a.E) ? a.b_router[e] : 0.f);
  }
  __syncthreads();
}

// Fused combine: the down projection adds both expert outputs into out, so this CTA's token rows
// start at zero.  Issued before the logits work, the stores drain while the loads wait on memory.
__device__ __forceinline__ void zero_out_rows(const RouterArgs& a, int chunk_t0, int valid) {
  if (a.zero_out == nullptr) return;
  const int n4 = a.d / 4;
  float4* o = reinterpret_cast<float4*>(a.zero_out + (size_t)chunk_t0 * a.d);
  for (int i = threadIdx.x; i < valid * n4; i += kRouterThreads) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// fp32 layers: FMA dot products with W_r staged in shared memory.
template <typename Tin, int EMAX>
__global__ void __launch_bounds__(kRouterThreads) router_top2_kernel(RouterArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  constexpr int VEC = Vec<Tin>::N;
  constexpr int SPAN = 32 * VEC;                // columns one warp covers per iteration
  constexpr int NW = kRouterThreads / 32;       // warps per CTA
  Tin* wsm = reinterpret_cast<Tin*>(smem_raw);
  __shared__ int s_idx[kRouterChunk][kMaxSlots];
  __shared__ float s_part[NW][4][EMAX];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_t0 = blockIdx.x * kRouterChunk;
  const int T = a.T, d = a.d, E = a.E;
  const int valid = min(kRouterChunk, T - chunk_t0);
  // Warps = G token groups (4 tokens each, the groups this chunk needs, rounded up to a power of
  // two) x S slices of the hidden dimension.  A full chunk gives G = 8, S = 1; a lone token gives
  // G = 1 and all 8 warps share its row, so small batches are not one warp's serial latency.
  const int need = (valid + 3) >> 2;
  const int G = need <= 1 ? 1 : (need <= 2 ? 2 : (need <= 4 ? 4 : 8));
  const int S = NW / G;
  const int g = warp % G, sl = warp / G;
  const int t0 = chunk_t0 + g * 4;
  const Tin* __restrict__ x = static_cast<const Tin*>(a.x);
  const Tin* __restrict__ w = static_cast<const Tin*>(a.w_router);
  pdl_trigger();
  pdl_wait();  // x may come from the previous kernel; the workspace from the previous forward
  zero_out_rows(a, chunk_t0, valid);

  float acc[4][EMAX];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[k][e] = 0.f;

  for (int d0 = 0; d0 < d; d0 += a.dchunk) {
    const int dc = min(a.dchunk, d - d0);
    __syncthreads();
    // stage W_r[:, d0 : d0 + dc]: eight independent 16-byte loads in flight per thread
    const int nvec = dc / VEC, total = E * nvec;
    for (int base = threadIdx.x; base < total; base += kRouterThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kRouterThreads;
        if (i < total) {
          const int e = i / nvec, jv = i - e * nvec;
          v[u] = __ldg(reinterpret_cast<const uint4*>(w + (size_t)e * d + d0 + jv * VEC));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kRouterThreads;
        if (i < total) {
          const int e = i / nvec, jv = i - e * nvec;
          *reinterpret_cast<uint4*>(wsm + (size_t)e * a.dchunk + jv * VEC) = v[u];
        }
      }
    }
    __syncthreads();
    const int n_it = (dc + SPAN - 1) / SPAN;
    const int it0 = (n_it * sl) / S, it1 = (n_it * (sl + 1)) / S;
    for (int it = it0; it < it1; it += 2) {
      // both iterations' token vectors are requested before any is used
      uint4 xr[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = (it + u) * SPAN + lane * VEC;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xr[u][k] = make_uint4(0u, 0u, 0u, 0u);
          if (it + u < it1 && j < dc && t0 + k < T)
            xr[u][k] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + k) * d + d0 + j));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int j = (it + u) * SPAN + lane * VEC;
        if (it + u < it1 && j < dc) {
          float xv[4][VEC];
#pragma unroll
          for (int k = 0; k < 4; ++k) Vec<Tin>::from_raw(xr[u][k], xv[k]);
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
    }
  }

  // warp all-reduce, then the S slices of each token group summed in slice order via shared memory
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[k][e] += __shfl_xor_sync(0xffffffffu, acc[k][e], o);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) s_part[warp][k][e] = acc[k][e];
  }
  __syncthreads();

  if (sl == 0 && lane < 4) {
    const int k = lane;
    const int t = t0 + k;
    float L[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      float v = s_part[g][k][e];
      for (int q = 1; q < S; ++q) v += s_part[g + q * G][k][e];
      L[e] = v + ((a.b_router != nullptr && e < E) ? a.b_router[e] : 0.f);
    }
    topk_store<EMAX>(a, L, t, s_idx[g * 4 + k]);
  }
  __syncthreads();
  finish_chunk(a, s_idx, valid, chunk_t0);
}


// bf16 layers: the logits GEMM on tensor cores with mma.sync m16n8k16 (bf16 x bf16 -> fp32).  Each
// warp owns 16 tokens x (8 * NT) experts over one slice of the hidden dimension; A fragments come
// straight from x in global memory (every 32-byte sector a warp touches is used whole), B fragments
// from W_r through L1/L2.  Partial tiles of the slices are summed in slice order in shared memory.
template <int NT>
__global__ void __launch_bounds__(kRouterThreads, 2) router_top2_mma_kernel(RouterArgs a) {
  constexpr int NW = kRouterThreads / 32;
  constexpr int EMAX = 8 * NT;
  constexpr int UNR = NT == 1 ? 8 : 4;  // 32-column blocks in flight per warp
  __shared__ float s_part[NW][16][EMAX];
  __shared__ int s_idx[kRouterChunk][kMaxSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_t0 = blockIdx.x * kRouterChunk;
  const int T = a.T, d = a.d, E = a.E;
  const int valid = min(kRouterChunk, T - chunk_t0);
  const int H = valid > 16 ? 2 : 1;  // 16-token halves with work
  const int S = NW / H;              // slices of the hidden dimension
  const int h = warp % H, sl = warp / H;
  const int g = lane >> 2, q = lane & 3;
  const int r0 = chunk_t0 + 16 * h;
  const bool v0 = r0 + g < T, v1 = r0 + g + 8 < T;
  const uint32_t* x0 = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                          (size_t)(v0 ? r0 + g : 0) * d);
  const uint32_t* x1 = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.x) +
                                                          (size_t)(v1 ? r0 + g + 8 : 0) * d);
  const uint32_t* wr[NT];
  bool wv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    wv[nt] = nt * 8 + g < E;
    wr[nt] = reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(a.w_router) +
                                               (size_t)(wv[nt] ? nt * 8 + g : 0) * d);
  }
  // k is summed over, so any permutation of it applied to A and B alike gives the same product.  Per
  // 32-column block, lane (g, q) loads columns 8q..8q+7 of its rows as one 16-byte vector and uses
  // them as logical k {2q, 2q+1, 2q+8, 2q+9} of two consecutive k-steps: one load instruction per row
  // per two MMAs, each instruction reading 64 contiguous bytes of 8 rows.
  const int nblk = d / 32;
  const int kb0 = (nblk * sl) / S, kb1 = (nblk * (sl + 1)) / S;
  pdl_trigger();
  pdl_wait();  // x may come from the previous kernel; the workspace from the previous forward
  zero_out_rows(a, chunk_t0, valid);
  // one bulk L2 prefetch per token row of this warp's column range: only the first round of fragment
  // loads below waits on HBM, the later rounds hit L2
  if (lane < 16 && kb1 > kb0) {
    const int row = r0 + lane;
    if (row < T) {
      const char* p = reinterpret_cast<const char*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)row * d +
                                                    (size_t)kb0 * 32);
      const uint32_t bytes = static_cast<uint32_t>(kb1 - kb0) * 64u;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
    }
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  for (int kb = kb0; kb < kb1; kb += UNR) {
    uint4 A0[UNR], A1[UNR], B[UNR][NT];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int vi = 4 * (kb + u) + q;  // 16-byte vector holding columns 32*(kb+u) + 8q .. +7
      const bool in = kb + u < kb1;
      A0[u] = (in && v0) ? __ldg(reinterpret_cast<const uint4*>(x0) + vi) : make_uint4(0u, 0u, 0u, 0u);
      A1[u] = (in && v1) ? __ldg(reinterpret_cast<const uint4*>(x1) + vi) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        B[u][nt] = (in && wv[nt]) ? __ldg(reinterpret_cast<const uint4*>(wr[nt]) + vi) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (kb + u < kb1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          // k-step 0 of the block: words x/y; k-step 1: words z/w
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0[u].x), "r"(A1[u].x), "r"(A0[u].y), "r"(A1[u].y), "r"(B[u][nt].x), "r"(B[u][nt].y));
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0[u].z), "r"(A1[u].z), "r"(A0[u].w), "r"(A1[u].w), "r"(B[u][nt].z), "r"(B[u][nt].w));
        }
      }
    }
  }
  // D fragment: acc[nt][0..1] = rows g, experts nt*8 + 2q, +1; acc[nt][2..3] = row g + 8
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s_part[warp][g][nt * 8 + 2 * q] = acc[nt][0];
    s_part[warp][g][nt * 8 + 2 * q + 1] = acc[nt][1];
    s_part[warp][g + 8][nt * 8 + 2 * q] = acc[nt][2];
    s_part[warp][g + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  __shared__ float s_logit[kRouterChunk][EMAX];
  sum_slices<EMAX>(a, s_part, s_logit, H, S, valid);
  if (threadIdx.x < valid) {
    float L[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) L[e] = s_logit[threadIdx.x][e];
    topk_store<EMAX>(a, L, chunk_t0 + threadIdx.x, s_idx[threadIdx.x]);
  }
  __syncthreads();
  finish_chunk(a, s_idx, valid, chunk_t0);
}

// Small and medium batches (up to 32 chunks of 32 tokens): the hidden dimension is split over kRsSplit
// CTAs per chunk, so every warp's fragment loads fit in one round (a single CTA would need four
// dependent rounds of HBM loads).  Each CTA sums its warps' slices in order and stores its partial
// logits; the CTA that finishes a chunk's split last (a per-chunk ticket, reset by that CTA) sums the
// kRsSplit partials in split order -- deterministic -- and does the top-k and the histogram.
constexpr int kRsSplit = 8;

template <int NT>
__global__ void __launch_bounds__(kRouterThreads, 2) router_split_kernel(RouterArgs a) {
  constexpr int NW = kRouterThreads / 32;
  constexpr int EMAX = 8 * NT;
  __shared__ float s_part[NW][16][EMAX];
  __shared__ int s_idx[kRouterChunk][kMaxSlots];
  __shared__ int s_lastsplit;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x / kRsSplit, split = blockIdx.x % kRsSplit;
  const int nchunks = gridDim.x / kRsSplit;
  const int chunk_t0 = chunk * kRouterChunk;
  const int T = a.T, d = a.d, E = a.E;
  const int valid = min(kRouterChunk, T - chunk_t0);
  const int H = valid > 16 ? 2 : 1;
  const int S = NW / H;
  const int h = warp % H, sl = warp / H;
  const int g = lane >> 2, q = lane & 3;
  const int r0 = chunk_t0 + 16 * h;
  const bool v0 = r0 + g < T, v1 = r0 + g + 8 < T;
  const uint4* x0 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)(v0 ? r0 + g : 0) * d);
  const uint4* x1 =
      reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)(v1 ? r0 + g + 8 : 0) * d);
  const uint4* wr[NT];
  bool wv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    wv[nt] = nt * 8 + g < E;
    wr[nt] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w_router) +
                                            (size_t)(wv[nt] ? nt * 8 + g : 0) * d);
  }
  // this CTA's 32-column blocks, then this warp's share of them
  const int nblk = d / 32;
  const int cb0 = (nblk * split) / kRsSplit, cb1 = (nblk * (split + 1)) / kRsSplit;
  const int kb0 = cb0 + ((cb1 - cb0) * sl) / S, kb1 = cb0 + ((cb1 - cb0) * (sl + 1)) / S;
  pdl_trigger();
  pdl_wait();  // x may come from the previous kernel; the workspace from the previous forward
  {
    // clearing out (when asked): this split's share of the chunk's rows
    const int r0s = (kRouterChunk * split) / kRsSplit, r1s = min((kRouterChunk * (split + 1)) / kRsSplit, valid);
    if (r1s > r0s) zero_out_rows(a, chunk_t0 + r0s, r1s - r0s);
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  constexpr int UNR = 8;
  for (int kb = kb0; kb < kb1; kb += UNR) {
    uint4 A0[UNR], A1[UNR], B[UNR][NT];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int vi = 4 * (kb + u) + q;
      const bool in = kb + u < kb1;
      A0[u] = (in && v0) ? __ldg(x0 + vi) : make_uint4(0u, 0u, 0u, 0u);
      A1[u] = (in && v1) ? __ldg(x1 + vi) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) B[u][nt] = (in && wv[nt]) ? __ldg(wr[nt] + vi) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      if (kb + u < kb1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0[u].x), "r"(A1[u].x), "r"(A0[u].y), "r"(A1[u].y), "r"(B[u][nt].x), "r"(B[u][nt].y));
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0[u].z), "r"(A1[u].z), "r"(A0[u].w), "r"(A1[u].w), "r"(B[u][nt].z), "r"(B[u][nt].w));
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s_part[warp][g][nt * 8 + 2 * q] = acc[nt][0];
    s_part[warp][g][nt * 8 + 2 * q + 1] = acc[nt][1];
    s_part[warp][g + 8][nt * 8 + 2 * q] = acc[nt][2];
    s_part[warp][g + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  // this split's partial logits of the chunk's 32 rows, warps' slices summed in order
  float* part = a.split_part + ((size_t)chunk * kRsSplit + split) * kRouterChunk * EMAX;
  for (int i = threadIdx.x; i < kRouterChunk * EMAX; i += blockDim.x) {
    const int r = i / EMAX, e = i - r * EMAX, hh = r / 16, rr = r - 16 * hh;
    float v = 0.f;
    if (hh < H) {
      v = s_part[hh][rr][e];
      for (int w = 1; w < S; ++w) v += s_part[hh + w * H][rr][e];
    }
    part[i] = v;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned before = atomicAdd(&a.sched->split_ticket[chunk], 1u);
    s_lastsplit = before == kRsSplit - 1;
    if (s_lastsplit) a.sched->split_ticket[chunk] = 0;  // ready for the next forward
  }
  __syncthreads();
  if (!s_lastsplit) {
    // fused dispatch: this CTA copies its own columns of the chunk's rows once all chunks are routed
    if (a.xp) fused_dispatch<2>(a, chunk, nchunks, chunk_t0, valid, nullptr, nullptr, cb0 * 32, cb1 * 32, false);
    return;
  }
  __threadfence();
  // every thread sums (row, expert) logits over the splits in split order, into s_part's space
  float(*s_logit)[EMAX] = reinterpret_cast<float(*)[EMAX]>(&s_part[0][0][0]);
  const float* base = a.split_part + (size_t)chunk * kRsSplit * kRouterChunk * EMAX;
  for (int i = threadIdx.x; i < kRouterChunk * EMAX; i += blockDim.x) {
    float p[kRsSplit];
#pragma unroll
    for (int sp = 0; sp < kRsSplit; ++sp) p[sp] = __ldcg(base + (size_t)sp * kRouterChunk * EMAX + i);
    float v = p[0];
#pragma unroll
    for (int sp = 1; sp < kRsSplit; ++sp) v += p[sp];
    const int e = i % EMAX;
    s_logit[i / EMAX][e] = v + ((a.b_router != nullptr && e < E) ? a.b_router[e] : 0.f);
  }
  __syncthreads();
  if (threadIdx.x < kRouterChunk) {
    float L[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) L[e] = s_logit[threadIdx.x][e];
    topk_store<EMAX>(a, L, chunk_t0 + threadIdx.x, s_idx[threadIdx.x]);
  }
  __syncthreads();
  __shared__ int s_rank[kRouterChunk * kMaxSlots];
  finish_chunk(a, s_idx, valid, chunk_t0, chunk, nchunks, a.xp ? s_rank : nullptr);
  if (a.xp) fused_dispatch<2>(a, chunk, nchunks, chunk_t0, valid, s_rank, s_idx, cb0 * 32, cb1 * 32, true);
}

// Large batches: the same logits GEMM with x streamed through shared memory by TMA.  The CTA's 32
// token rows arrive in stages of 512 columns (eight 64-column boxes, 128-byte swizzle: 1 KB of
// every row at a time, which DRAM serves better than shorter pieces) in a kRtStages-deep ring, so
// the copy engine keeps 96 KB per CTA in flight whatever the warps do;
// warp (h, sl) multiplies the 16 rows of half h over its share of each stage's eight 32-column
// blocks (fragments read from the swizzled rows without bank conflicts), W_r fragments come from
// L1/L2 one stage ahead in registers.  Each warp sums its blocks stage by stage (a fixed order), the
// warps' partial tiles are summed in slice order in shared memory; top-k and the histogram as above.
constexpr int kRtStages = 3;
constexpr int kRtCols = 512;                                 // columns per stage (1 KB of every row)
constexpr int kRtBlk = kRtCols / 32;                         // 32-column blocks per stage
constexpr int kRtStageBytes = kRouterChunk * kRtCols * 2;    // 32 KB
constexpr int kRtSmem = 1024 + kRtStages * kRtStageBytes + 2 * kRtStages * 8;

__device__ __forceinline__ uint32_t rt_smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool rt_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok = 0;
  uint64_t t0 = 0;
  for (int spin = 0;; ++spin) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    uint64_t now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    if (spin == 0) t0 = now;
    else if (now - t0 > 2000000000ull) return false;  // 2 s: the copy engine never delivered
  }
}

template <int NT>
__global__ void __launch_bounds__(kRouterThreads, 2)
    router_tma_kernel(const __grid_constant__ CUtensorMap tmx, RouterArgs a) {
  constexpr int NW = kRouterThreads / 32;
  constexpr int EMAX = 8 * NT;
  extern __shared__ __align__(1024) uint8_t rt_raw[];
  uint8_t* stg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rt_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg + kRtStages * kRtStageBytes);
  const uint32_t full0 = rt_smem_u32(bars), empty0 = rt_smem_u32(bars + kRtStages);
  __shared__ float s_part[NW][16][EMAX];
  __shared__ int s_idx[kRouterChunk][kMaxSlots];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk_t0 = blockIdx.x * kRouterChunk;
  const int T = a.T, d = a.d, E = a.E;
  const int valid = min(kRouterChunk, T - chunk_t0);
  const int H = valid > 16 ? 2 : 1;  // 16-token halves with work
  const int S = NW / H;              // warps sharing a half: each takes 8 / S blocks of a stage
  const int h = warp % H, sl = warp / H;
  const int g = lane >> 2, q = lane & 3;
  const int j0 = (kRtBlk * sl) / S, j1 = (kRtBlk * (sl + 1)) / S;  // this warp's blocks of each stage
  constexpr int kJ = kRtBlk / 4;  // most blocks a warp takes per stage (4 or more warps share a half)
  const int nst = d / kRtCols;
  const uint4* wr[NT];
  bool wv[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    wv[nt] = nt * 8 + g < E;
    wr[nt] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.w_router) +
                                            (size_t)(wv[nt] ? nt * 8 + g : 0) * d);
  }
  if (threadIdx.x == 0) {
    for (int st = 0; st < kRtStages; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(full0 + 8 * st), "r"(1) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty0 + 8 * st), "r"(NW) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // x may come from the previous kernel; the workspace from the previous forward
  zero_out_rows(a, chunk_t0, valid);
  auto issue = [&](int st) {  // thread 0: stage st into slot st % kRtStages
    const int slot = st % kRtStages;
    const uint32_t fb = full0 + 8 * slot;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(kRtStageBytes) : "memory");
#pragma unroll
    for (int b = 0; b < kRtCols / 64; ++b)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
          "[%4];" ::"r"(rt_smem_u32(stg + slot * kRtStageBytes + b * 4096)),
          "l"(reinterpret_cast<uint64_t>(&tmx)), "r"(st * kRtCols + b * 64), "r"(chunk_t0), "r"(fb)
          : "memory");
  };
  if (threadIdx.x == 0)
    for (int st = 0; st < kRtStages && st < nst; ++st) issue(st);

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  // W_r fragments of this warp's blocks, one stage ahead
  uint4 Bn[kJ][NT];
  auto load_b = [&](int st) {
#pragma unroll
    for (int u = 0; u < kJ; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int j = j0 + u;
        Bn[u][nt] = (j < j1 && wv[nt]) ? __ldg(wr[nt] + 4 * (st * kRtBlk + j) + q) : make_uint4(0u, 0u, 0u, 0u);
      }
  };
  load_b(0);
  bool ok = true;
  const int r_lo = 16 * h + g, r_hi = r_lo + 8;  // rows of this lane inside the CTA's 32
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kRtStages;
    const uint32_t par = static_cast<uint32_t>((st / kRtStages) & 1);
    uint4 B[kJ][NT];
#pragma unroll
    for (int u = 0; u < kJ; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) B[u][nt] = Bn[u][nt];
    if (st + 1 < nst) load_b(st + 1);
    if (ok && !rt_wait(full0 + 8 * slot, par)) {
      ok = false;
      atomicOr(&a.sched->status, kStatusTimeoutRouter);
    }
    const uint8_t* sb = stg + slot * kRtStageBytes;
#pragma unroll
    for (int u = 0; u < kJ; ++u) {
      const int j = j0 + u;
      if (j < j1) {
        // block j: box j / 2, 16-byte chunk 4 * (j % 2) + q of the row, swizzled by row % 8
        const int c = 4 * (j & 1) + q;
        const uint8_t* box = sb + (j >> 1) * 4096;
        const uint4 A0 = *reinterpret_cast<const uint4*>(box + r_lo * 128 + ((c ^ (r_lo & 7)) << 4));
        const uint4 A1 = *reinterpret_cast<const uint4*>(box + r_hi * 128 + ((c ^ (r_hi & 7)) << 4));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0.x), "r"(A1.x), "r"(A0.y), "r"(A1.y), "r"(B[u][nt].x), "r"(B[u][nt].y));
          asm volatile(
              "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};"
              : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
              : "r"(A0.z), "r"(A1.z), "r"(A0.w), "r"(A1.w), "r"(B[u][nt].z), "r"(B[u][nt].w));
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * slot) : "memory");
    if (threadIdx.x == 0 && st + kRtStages < nst) {
      // the slot is refilled once all warps have read it
      if (ok && !rt_wait(empty0 + 8 * slot, par)) {
        ok = false;
        atomicOr(&a.sched->status, kStatusTimeoutRouter);
      }
      if (ok) issue(st + kRtStages);
    }
  }
  // every copy issued has landed before the CTA may leave (bounded)
  if (threadIdx.x == 0)
    for (int st = nst - kRtStages > 0 ? nst - kRtStages : 0; st < nst; ++st)
      rt_wait(full0 + 8 * (st % kRtStages), static_cast<uint32_t>((st / kRtStages) & 1));
  // D fragment: acc[nt][0..1] = rows g, experts nt*8 + 2q, +1; acc[nt][2..3] = row g + 8
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s_part[warp][g][nt * 8 + 2 * q] = acc[nt][0];
    s_part[warp][g][nt * 8 + 2 * q + 1] = acc[nt][1];
    s_part[warp][g + 8][nt * 8 + 2 * q] = acc[nt][2];
    s_part[warp][g + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  // the summed logits go to the first ring slot: every stage has landed and been read
  float(*s_logit)[EMAX] = reinterpret_cast<float(*)[EMAX]>(stg);
  sum_slices<EMAX>(a, s_part, s_logit, H, S, 16 * H);
  if (threadIdx.x < 16 * H) {
    float L[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) L[e] = s_logit[threadIdx.x][e];
    topk_store<EMAX>(a, L, chunk_t0 + threadIdx.x, s_idx[threadIdx.x]);
  }
  __syncthreads();
  finish_chunk(a, s_idx, valid, chunk_t0);
}

// Cooperative launch (every CTA resident: the fused dispatch's grid barrier), with programmatic
// dependent launch like the other kernels.
template <typename... KArgs, typename... Args>
cudaError_t coop_launch(void (*kernel)(KArgs...), int grid, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int resident_per_sm(const void* kernel, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kRouterThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm;
}

template <typename Tin, int EMAX>
cudaError_t launch_router_t(const RouterArgs& a, int nchunks, cudaStream_t s) {
  const int smem = EMAX * a.dchunk * (int)sizeof(Tin);
  return pdl_launch(router_top2_kernel<Tin, EMAX>, dim3(nchunks), dim3(kRouterThreads), smem, s, a);
}

template <typename Tin, int EMAX>
cudaError_t prepare_router_t() {
  return cudaFuncSetAttribute(router_top2_kernel<Tin, EMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRouterMaxSmem);
}

}  // namespace

cudaError_t prepare_router(int dtype, int E) {
  if (dtype != 0) {
    cudaError_t e = cudaFuncSetAttribute(router_tma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(router_tma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e != cudaSuccess) return e;
  }
  if (dtype == 0) return E <= 4 ? prepare_router_t<float, 4>() : E <= 8 ? prepare_router_t<float, 8>()
                                                                       : prepare_router_t<float, 16>();
  return E <= 4 ? prepare_router_t<__nv_bfloat16, 4>() : E <= 8 ? prepare_router_t<__nv_bfloat16, 8>()
                                                                 : prepare_router_t<__nv_bfloat16, 16>();
}

int router_smem_bytes(int dtype, int E, int dchunk) {
  const int emax = E <= 4 ? 4 : (E <= 8 ? 8 : 16);
  return emax * dchunk * (dtype == 0 ? 4 : 2);
}

int router_tma_cols() { return kRtCols; }

// bf16, d a multiple of router_tma_cols(); tmx maps x [T, d] with 64 x 32 boxes, 128-byte swizzle
cudaError_t launch_router_tma(const CUtensorMap& tmx, const RouterArgs& a, int nchunks, cudaStream_t s) {
  if (a.E <= 8) return pdl_launch(router_tma_kernel<1>, dim3(nchunks), dim3(kRouterThreads), kRtSmem, s, tmx, a);
  return pdl_launch(router_tma_kernel<2>, dim3(nchunks), dim3(kRouterThreads), kRtSmem, s, tmx, a);
}

// bf16, at most kRouterSplitMaxChunks chunks, d a multiple of 32 * kRsSplit; a.split_part holds
// [nchunks][kRsSplit][32][EMAX] floats
cudaError_t launch_router_split(const RouterArgs& a, int nchunks, cudaStream_t s) {
  if (a.E <= 8) return pdl_launch(router_split_kernel<1>, dim3(nchunks * kRsSplit), dim3(kRouterThreads), 0, s, a);
  return pdl_launch(router_split_kernel<2>, dim3(nchunks * kRsSplit), dim3(kRouterThreads), 0, s, a);
}
int router_split_factor() { return kRsSplit; }

cudaError_t launch_router_split_fused(const RouterArgs& a, int nchunks, cudaStream_t s) {
  if (a.E <= 8) return coop_launch(router_split_kernel<1>, nchunks * kRsSplit, 0, s, a);
  return coop_launch(router_split_kernel<2>, nchunks * kRsSplit, 0, s, a);
}

int router_split_fused_max_chunks(int E, int num_sms) {
  const void* k = E <= 8 ? reinterpret_cast<const void*>(router_split_kernel<1>)
                         : reinterpret_cast<const void*>(router_split_kernel<2>);
  return resident_per_sm(k, 0) * num_sms / kRsSplit;
}

cudaError_t launch_router(int dtype, const RouterArgs& a, int nchunks, cudaStream_t s) {
  if (dtype == 0) {
    if (a.E <= 4) return launch_router_t<float, 4>(a, nchunks, s);
    if (a.E <= 8) return launch_router_t<float, 8>(a, nchunks, s);
    return launch_router_t<float, 16>(a, nchunks, s);
  }
  if (a.d % 32 == 0) {
    if (a.E <= 8) return pdl_launch(router_top2_mma_kernel<1>, dim3(nchunks), dim3(kRouterThreads), 0, s, a);
    return pdl_launch(router_top2_mma_kernel<2>, dim3(nchunks), dim3(kRouterThreads), 0, s, a);
  }
  if (a.E <= 4) return launch_router_t<__nv_bfloat16, 4>(a, nchunks, s);
  if (a.E <= 8) return launch_router_t<__nv_bfloat16, 8>(a, nchunks, s);
  return launch_router_t<__nv_bfloat16, 16>(a, nchunks, s);
}

}  // namespace colibri
