// Grouped expert GEMM with the operands swapped ("weight-major"), on CTA pairs (tcgen05 cta_group::2):
// the expert's weight rows on the MMA's M side (256 per pair, 128 per CTA) and its token rows on N.
//
// Same computation as gemm_tcgen05_2sm.cu (the Compute stage of zskr.cn/news/2272131, "Colibri: a
// lightweight C MoE inference engine for edge devices", 2.1: one GEMM per expert over its contiguous
// rows, the activation fused in the epilogue as in m.nxbn.cn/news/48047 2.1), for layers whose
// experts hold few rows (about 256 or fewer).  There the CTA-pair kernel pads each expert's rows to
// 256-row tiles and spends half of every ring stage on token rows, so each SM keeps only 96 KB of
// weights in flight; a weight-streaming GEMM runs at (weight bytes in flight) / (memory latency).
// Here a work item is (expert e, 256-row weight tile w, token tile t of at most NT rows):
//
//   - N = the tile's token count rounded up to 32 (at most NT, host-chosen per launch); each CTA
//     stages 16 KB of weights and N/2 token rows (64 N bytes) per 64-wide K step, so NT = 160 gives
//     seven stages and 112 KB of weights in flight per SM, NT = 128 eight stages and 128 KB;
//   - the leader CTA issues tcgen05.mma.cta_group::2 (M=256, N, K=16): CTA c's accumulator holds its
//     128 weight rows (TMEM lanes) x the tile's N tokens (columns);
//   - SwiGLU: CTA c's weight tile is the gate rows of hidden units 128 w + 64 c + [0, 64) (arena
//     rows 256 w + 64 c + [0, 64)) and their up rows (128 further on), two 64-row boxes, so TMEM
//     lanes l and l + 64 hold the gate and up value of the same hidden unit; the warps holding the
//     up values hand them to the warps holding the gates through shared memory;
//   - every epilogue turns its 32 x 32 chunks around in shared memory, so that a thread writes 16
//     bytes of one output row (H rows in bf16, Y rows or the gate-weighted fp32 sum into out).
//
// Items are handed out in index order at run time (a counter shared by all pairs, a per-pair id
// queue), token tiles of one weight tile adjacent, so that the pairs reading the same weight tile
// run together.  Waits are bounded (a status bit and an orderly exit when one runs out); TMEM is
// allocated and freed collectively by one warp of each CTA.
//
// Fused form (both projections in one launch): the up projection's items come first, then the down
// projection's.  A pair that runs out of up items goes straight on to down items instead of idling
// through the up projection's last wave and a second launch.  A down item of expert e reads H rows
// of e that other pairs wrote: every epilogue warp of an up item fences its H stores for the async
// proxy and adds 1 to wm_done[e] with a gpu-scope release once they are out, and the producer of a
// down item waits (acquire, bounded) until wm_done[e] counts all 8 warps of all of e's up items.  The
// fp32 output the down projection adds into is cleared by the clearing warps, which count themselves
// in wm_cleared; the combine epilogue waits for all of them before its first addition.  Every item,
// the first included, comes from the shared counter, so a pair only ever waits for up items that
// running pairs hold: no co-residency assumption beyond the pair itself.
#include "tcgen05_ptx.cuh"

namespace colibri {
namespace {

using namespace ptx;

constexpr int WBM = 128, WBK = 64, WUMMA_K = 16;
constexpr int WA_BYTES = WBM * WBK * 2;  // 16 KB of weight rows per CTA per K step
constexpr int WRING_BYTES = 192 * 1024;
constexpr int WSTAGES_MAX = 12;
constexpr int WNUM_THREADS = 192;
constexpr int WNUM_THREADS_ZERO = 192 + 32 * kZeroWarps;
constexpr uint32_t WTMEM_COLS = 512;  // two accumulators of up to 256 token columns
constexpr int WTQ = 4;                // item-id queue depth
constexpr int kWPublishAt = 4;        // K step of an item at which the leader hands out the next id
constexpr int WSTG_LD = 36;           // staging row stride in words (16-byte aligned rows)
constexpr int WSTG_BYTES = 4 * 32 * WSTG_LD * 4;
// full, empty, tmem_full[2], tmem_empty[2], drain, item queue full / empty
constexpr int WNUM_BARS = 2 * WSTAGES_MAX + 5 + 2 * WTQ;
// + counts, offsets, token tiles, items before each expert (two projections), the item queue
constexpr int WSMEM_BYTES =
    1024 + WRING_BYTES + WSTG_BYTES + WNUM_BARS * 8 + 16 + 4 * (5 * kMaxE + 4 + WTQ);
static_assert(WSMEM_BYTES <= 227 * 1024, "weight-major GEMM shared memory");

struct WmCoord {
  int e, w, t;
};

// Item p -> (expert, weight tile, token tile); istart[e] = items before expert e, tt[e] = its token tiles.
__device__ __forceinline__ WmCoord decode_wm(int p, const int* istart, const int* tt, int E) {
  int e = 0;
  while (e + 1 < E && istart[e + 1] <= p) ++e;
  const int local = p - istart[e];
  WmCoord c;
  c.e = e;
  c.w = local / tt[e];
  c.t = local - c.w * tt[e];
  return c;
}

__device__ __forceinline__ void wm_pair_sync(int q) {
  if (q & 1)
    asm volatile("bar.sync 3, 64;" ::: "memory");
  else
    asm volatile("bar.sync 2, 64;" ::: "memory");
}

template <int EPI>
__device__ __forceinline__ void wm_epilogue(const GemmArgs& a, const WmCoord& c, int row0, int nreal, int n,
                                            uint32_t tbase, int q, int lane, int rank, uint32_t* s_stage) {
  uint32_t* stg = s_stage + q * (32 * WSTG_LD);
  const int nch = n / 32;
  if constexpr (EPI == kEpiSwiGLU) {
    // warps 0, 1: gate values of hidden units 64 rank + 32 q + lane; warps 2, 3: their up values
    const int f0 = c.w * WBM + 64 * rank + 32 * (q & 1);  // this warp pair's units
    const uint32_t* stg_up = s_stage + (q | 2) * (32 * WSTG_LD) + lane * WSTG_LD;
    __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + ch * 32, v);
      if (q >= 2) {
        uint4* dst = reinterpret_cast<uint4*>(stg + lane * WSTG_LD);
#pragma unroll
        for (int w4 = 0; w4 < 8; ++w4) dst[w4] = make_uint4(v[4 * w4], v[4 * w4 + 1], v[4 * w4 + 2], v[4 * w4 + 3]);
        wm_pair_sync(q);  // up values in place
        wm_pair_sync(q);  // taken by the gate warp
      } else {
        wm_pair_sync(q);
        float h[32];
#pragma unroll
        for (int w4 = 0; w4 < 8; ++w4) {
          const uint4 u = reinterpret_cast<const uint4*>(stg_up)[w4];
          h[4 * w4] = silu_fast(__uint_as_float(v[4 * w4])) * __uint_as_float(u.x);
          h[4 * w4 + 1] = silu_fast(__uint_as_float(v[4 * w4 + 1])) * __uint_as_float(u.y);
          h[4 * w4 + 2] = silu_fast(__uint_as_float(v[4 * w4 + 2])) * __uint_as_float(u.z);
          h[4 * w4 + 3] = silu_fast(__uint_as_float(v[4 * w4 + 3])) * __uint_as_float(u.w);
        }
        wm_pair_sync(q);
        // transpose: token j's 32 hidden units in row j of this warp's staging tile
#pragma unroll
        for (int j = 0; j < 32; ++j) stg[j * WSTG_LD + lane] = __float_as_uint(h[j]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int idx = 32 * i + lane, j = idx >> 2, g8 = idx & 3;  // token j, units 8 g8 ..
          const uint4 lo = *reinterpret_cast<const uint4*>(stg + j * WSTG_LD + 8 * g8);
          const uint4 hi = *reinterpret_cast<const uint4*>(stg + j * WSTG_LD + 8 * g8 + 4);
          const int tj = 32 * ch + j;
          if (tj < nreal) {
            const uint4 pk = make_uint4(pack_bf16(__uint_as_float(lo.x), __uint_as_float(lo.y)),
                                        pack_bf16(__uint_as_float(lo.z), __uint_as_float(lo.w)),
                                        pack_bf16(__uint_as_float(hi.x), __uint_as_float(hi.y)),
                                        pack_bf16(__uint_as_float(hi.z), __uint_as_float(hi.w)));
            *reinterpret_cast<uint4*>(hout + static_cast<size_t>(row0 + tj) * a.ldo + f0 + 8 * g8) = pk;
          }
        }
        __syncwarp();  // the staging tile is rewritten next
      }
    }
  } else if constexpr (EPI == kEpiReluBias) {
    const int f0 = c.w * 2 * WBM + WBM * rank + 32 * q;  // this warp's 32 units
    const float b = a.bias[static_cast<size_t>(c.e) * a.out_cols + f0 + lane];
    __nv_bfloat16* hout = static_cast<__nv_bfloat16*>(a.out);
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) stg[j * WSTG_LD + lane] = __float_as_uint(fmaxf(__uint_as_float(v[j]) + b, 0.f));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = 32 * i + lane, j = idx >> 2, g8 = idx & 3;
        const uint4 lo = *reinterpret_cast<const uint4*>(stg + j * WSTG_LD + 8 * g8);
        const uint4 hi = *reinterpret_cast<const uint4*>(stg + j * WSTG_LD + 8 * g8 + 4);
        const int tj = 32 * ch + j;
        if (tj < nreal) {
          const uint4 pk = make_uint4(pack_bf16(__uint_as_float(lo.x), __uint_as_float(lo.y)),
                                      pack_bf16(__uint_as_float(lo.z), __uint_as_float(lo.w)),
                                      pack_bf16(__uint_as_float(hi.x), __uint_as_float(hi.y)),
                                      pack_bf16(__uint_as_float(hi.z), __uint_as_float(hi.w)));
          *reinterpret_cast<uint4*>(hout + static_cast<size_t>(row0 + tj) * a.ldo + f0 + 8 * g8) = pk;
        }
      }
      __syncwarp();
    }
  } else {
    // fp32 results of output columns d0 + lane: Y rows, or (kEpiCombineF32) out[token] +=
    // gate * (acc (+ b2)); with two slots and a zeroed output the two reductions give
    // RN(g0*y0 + g1*y1) in either order, the value the separate combine computes
    constexpr bool kCombine = EPI == kEpiCombineF32;
    const int d0 = c.w * 2 * WBM + WBM * rank + 32 * q;
    const float b = a.bias ? a.bias[static_cast<size_t>(c.e) * a.out_cols + d0 + lane] : 0.f;
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      uint32_t v[32];
      tmem_ld32_sync(tbase + ch * 32, v);
      // token and gate (or output row) of the chunk's token `lane`
      const int tl = 32 * ch + lane;
      const bool lv = tl < nreal;
      const int my_tok = kCombine && lv ? __ldcg(a.token_of_row + row0 + tl)
                                        : (!kCombine && a.row_map != nullptr && lv ? __ldcg(a.row_map + row0 + tl)
                                                                                    : row0 + tl);
      const float my_g = kCombine && lv ? __ldcg(a.gate_of_row + row0 + tl) : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float y = __uint_as_float(v[j]);
        if (a.bias) y += b;
        stg[j * WSTG_LD + lane] = __float_as_uint(y);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int idx = 32 * i + lane, j = idx >> 3, g4 = idx & 7;  // token j, columns 4 g4 ..
        const int tok = __shfl_sync(0xffffffffu, my_tok, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        const uint4 raw = *reinterpret_cast<const uint4*>(stg + j * WSTG_LD + 4 * g4);
        if (32 * ch + j < nreal) {
          float* o = static_cast<float*>(a.out) + static_cast<size_t>(tok) * a.ldo + d0 + 4 * g4;
          if constexpr (kCombine) {
            red_add_v4(o, __fmul_rn(g, __uint_as_float(raw.x)), __fmul_rn(g, __uint_as_float(raw.y)),
                       __fmul_rn(g, __uint_as_float(raw.z)), __fmul_rn(g, __uint_as_float(raw.w)));
          } else {
            *reinterpret_cast<uint4*>(o) = raw;
          }
        }
      }
      __syncwarp();
    }
  }
}

__device__ __forceinline__ uint32_t wm_ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void wm_red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void wm_fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Bounded wait until *p >= target (acquire); false once timeout_ns has passed or the CTA aborts.
__device__ __forceinline__ bool wm_wait_count(const uint32_t* p, uint32_t target, volatile int* abort,
                                              uint64_t timeout_ns) {
  if (wm_ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (wm_ld_acquire(p) < target) {
    if (*abort || globaltimer_ns() - t0 > timeout_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// EPI2 < 0: one projection (P.args[0], P.maps[0]).  EPI2 >= 0: the fused form, up (EPI) then down (EPI2).
template <int EPI, int EPI2>
__global__ void __launch_bounds__(WNUM_THREADS_ZERO, 1) tc_wm_gemm_kernel(const __grid_constant__ WmFused P) {
  constexpr bool FUSED = EPI2 >= 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const GemmArgs& a = P.args[0];                       // shared fields: sched, E, status, timeout, counter
  const int NT = a.wm_ntok;                            // token tile (multiple of 32, <= 256)
  const int stage_bytes = WA_BYTES + 64 * NT;          // weights + NT / 2 token rows of 128 bytes
  int nst = WRING_BYTES / stage_bytes;
  if (nst > WSTAGES_MAX) nst = WSTAGES_MAX;
  const int NS = nst;
  uint32_t* s_stage = reinterpret_cast<uint32_t*>(smem + WRING_BYTES);  // epilogue staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s_stage) + WSTG_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + WNUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_counts = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_offsets = s_counts + kMaxE;
  int* s_tt = s_offsets + kMaxE + 1;
  int* s_istart = s_tt + kMaxE + 1;             // [2][kMaxE + 1]: items before expert e, per projection
  volatile int* s_item = s_istart + 2 * (kMaxE + 1);  // item-id queue

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + WSTAGES_MAX);
  const uint32_t tfull0 = smem_u32(bars + 2 * WSTAGES_MAX);
  const uint32_t tempty0 = smem_u32(bars + 2 * WSTAGES_MAX + 2);
  const uint32_t drain = smem_u32(bars + 2 * WSTAGES_MAX + 4);
  const uint32_t tqf0 = smem_u32(bars + 2 * WSTAGES_MAX + 5);
  const uint32_t tqe0 = smem_u32(bars + 2 * WSTAGES_MAX + 5 + WTQ);
  const bool DYN = FUSED || a.tile_ctr != nullptr;
  const bool ALLDYN = FUSED;  // the first item from the counter too

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  Sched* const sched = const_cast<Sched*>(a.sched);

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < WSTAGES_MAX; ++s) {
      mbar_init(full0 + 8 * s, 1);   // leader's: one arrive with both CTAs' TMA bytes per phase
      mbar_init(empty0 + 8 * s, 1);  // each CTA's: one multicast commit per phase
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 8);  // leader's: 4 epilogue warps of each CTA
    }
    mbar_init(drain, 1);
    for (int i = 0; i < WTQ; ++i) {
      mbar_init(tqf0 + 8 * i, 1);
      mbar_init(tqe0 + 8 * i, 10);  // leader: MMA + 4 epilogue warps; peer: producer + 4 epilogue warps
    }
    *s_abort = 0;
    fence_mbar_init();
    for (int ph = 0; ph < (FUSED ? 2 : 1); ++ph) {
      prefetch_tmap(&P.maps[ph].w);
      for (int i = 0; i < kWmTokMaps; ++i) prefetch_tmap(&P.maps[ph].tok[i]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), WTMEM_COLS);
    tmem_relinquish_pair();
  }
  pdl_wait();  // the routing summary and the token rows come from earlier kernels
  if (a.clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.clear_word = 0u;
  if (threadIdx.x < kMaxE) s_counts[threadIdx.x] = threadIdx.x < E ? sched->counts[threadIdx.x] : 0;
  if (threadIdx.x < kMaxE + 1) s_offsets[threadIdx.x] = threadIdx.x <= E ? sched->offsets[threadIdx.x] : 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int ph = 0; ph < 2; ++ph) {
      const int n_w = P.args[FUSED ? ph : 0].n_per_expert / (2 * WBM);  // 256-row weight tiles per expert
      int acc = 0;
      for (int e = 0; e < E; ++e) {
        if (ph == 0) s_tt[e] = (s_counts[e] + NT - 1) / NT;
        s_istart[ph * (kMaxE + 1) + e] = acc;
        acc += n_w * s_tt[e];
      }
      s_istart[ph * (kMaxE + 1) + E] = acc;
    }
  }
  tc_fence_before();
  cluster_sync();  // barrier inits and TMEM addresses visible across the pair
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total0 = s_istart[E];
  const int total = FUSED ? total0 + s_istart[kMaxE + 1 + E] : total0;
  const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  // item p -> projection and coordinates; the token tile: first row, real rows, MMA width N (rows
  // rounded up to 32)
  auto item = [&](int p, int& ph, WmCoord& c, int& row0, int& nreal, int& n) {
    ph = FUSED && p >= total0 ? 1 : 0;
    c = decode_wm(p - (ph ? total0 : 0), s_istart + ph * (kMaxE + 1), s_tt, E);
    row0 = s_offsets[c.e] + c.t * NT;
    nreal = min(NT, s_counts[c.e] - c.t * NT);
    n = (nreal + 31) & ~31;
  };

  // Item order: (ALLDYN) every item, or (DYN) every item after pair i's first (item i), comes from a
  // counter shared by all pairs; the leader's producer takes it and hands it to the pair's other roles
  // through a WTQ-deep queue in both CTAs' shared memory.  Else pair i takes items i, i + n_pairs, ...
  struct Seq {
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
  };
  auto take = [&](Seq& sq, bool arrive) -> int {
    if (!mbar_wait_cluster(tqf0 + 8 * sq.slot, sq.ph, s_abort, a.timeout_ns)) {
      sq.ok = false;
      return -1;
    }
    const int p = s_item[sq.slot];
    if (arrive) {
      if (leader)
        mbar_arrive(tqe0 + 8 * sq.slot);
      else
        mbar_arrive_peer(mapa_shared(tqe0 + 8 * sq.slot, 0));
    }
    if (++sq.slot == WTQ) {
      sq.slot = 0;
      sq.ph ^= 1u;
    }
    return p;
  };
  auto seq_first = [&](Seq& sq, bool arrive) -> int {
    if (ALLDYN) return take(sq, arrive);
    return pair_id < total ? pair_id : -1;
  };
  auto seq_next = [&](Seq& sq, int p, bool arrive) -> int {
    if (DYN) return take(sq, arrive);
    p += n_pairs;
    return p < total ? p : -1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      Seq sq, pub;
      auto publish = [&](int p) -> bool {
        if (!mbar_wait(tqe0 + 8 * pub.slot, pub.ph ^ 1u, s_abort, a.timeout_ns)) return false;
        s_item[pub.slot] = p;
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(s_item + pub.slot)), 1), p);
        mbar_arrive(tqf0 + 8 * pub.slot);
        mbar_arrive_remote(mapa_shared(tqf0 + 8 * pub.slot, 1));  // release.cluster: the id is there
        if (++pub.slot == WTQ) {
          pub.slot = 0;
          pub.ph ^= 1u;
        }
        return true;
      };
      auto fetch = [&]() -> int {
        const int p = (ALLDYN ? 0 : n_pairs) + static_cast<int>(atomicAdd(a.tile_ctr, 1u));
        return p < total ? p : -1;
      };
      int p = -1, p_next = -1;
      if (ALLDYN) {
        if (leader) {
          p = fetch();
          ok = publish(p);
        } else {
          p = take(sq, true);
          ok = sq.ok;
        }
      } else {
        p = seq_first(sq, true);
      }
      for (; ok && p >= 0;) {
        int ph, row0, nreal, n;
        WmCoord c;
        item(p, ph, c, row0, nreal, n);
        const GemmArgs& ap = P.args[ph];
        const WmMaps& mp = P.maps[ph];
        const int num_kb = (ap.K + WBK - 1) / WBK;
        const int half_n = n / 2;
        const CUtensorMap* tm_tok = &mp.tok[half_n / 16 - 1];
        const int tok_row = row0 + static_cast<int>(rank) * half_n;
        const int wrow = c.e * ap.n_per_expert + c.w * 2 * WBM;
        const uint32_t stage_tx = 2u * static_cast<uint32_t>(WA_BYTES + 128 * half_n);
        const bool gated = ph == 0 && EPI == kEpiSwiGLU;  // gate / up halves in two 64-row boxes
        if (FUSED && ph == 1) {
          // H rows of expert e: every epilogue warp of every up item of e has released its stores
          const uint32_t need = 8u * static_cast<uint32_t>(P.args[0].n_per_expert / (2 * WBM)) * s_tt[c.e];
          if (!wm_wait_count(&sched->wm_done[c.e], need, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          wm_fence_proxy_async_global();  // the acquired H rows are read next by TMA
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t full_leader = mapa_shared(full0 + 8 * stage, 0);
          if (leader) {
            mbar_arrive_expect_tx(full0 + 8 * stage, stage_tx);
            armed |= 1u << stage;
            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          }
          const uint32_t sa = smem_u32(smem + stage * stage_bytes);
          if (gated) {
            // gate rows 256 w + 64 rank + [0, 64) and their up rows 128 further on
            tma_load_2d_pair(sa, &mp.w, full_leader, kb * WBK, wrow + 64 * static_cast<int>(rank));
            tma_load_2d_pair(sa + WA_BYTES / 2, &mp.w, full_leader, kb * WBK, wrow + WBM + 64 * static_cast<int>(rank));
          } else {
            tma_load_2d_pair(sa, &mp.w, full_leader, kb * WBK, wrow + WBM * static_cast<int>(rank));
          }
          tma_load_2d_pair(sa + WA_BYTES, tm_tok, full_leader, kb * WBK, tok_row);
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
          if (DYN && leader && kb == 0) p_next = fetch();
          if (DYN && leader && kb == (num_kb > kWPublishAt ? kWPublishAt : num_kb - 1)) {
            if (!publish(p_next)) {
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        if (DYN && leader) {
          p = p_next;
        } else {
          p = seq_next(sq, p, true);
          ok = sq.ok;
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
        *s_abort = 1;
      }
      // the leader's full barriers complete only when both CTAs' copies have landed
      for (int s = 0; s < NS; ++s)
        if (armed & (1u << s)) {
          volatile int never = 0;
          mbar_wait(full0 + 8 * s, (armed_phase >> s) & 1u, &never, a.timeout_ns);
        }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (leader only)
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      Seq sq;
      int p = seq_first(sq, true);
      bool ok = sq.ok;
      for (; ok && p >= 0; p = seq_next(sq, p, true), ok = ok && sq.ok) {
        int ph, row0, nreal, n;
        WmCoord c;
        item(p, ph, c, row0, nreal, n);
        const int num_kb = (P.args[ph].K + WBK - 1) / WBK;
        const uint32_t idesc = make_idesc_bf16(2 * WBM, n);
        if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_phase ^ 1u, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * 256);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * stage_bytes);
          const uint32_t b_addr = a_addr + WA_BYTES;
#pragma unroll
          for (int k = 0; k < WBK / WUMMA_K; ++k)
            umma_bf16_pair(d_tmem, sw128_desc(a_addr + k * WUMMA_K * 2), sw128_desc(b_addr + k * WUMMA_K * 2), idesc,
                           (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(empty0 + 8 * stage, 0x3);
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(tfull0 + 8 * acc, 0x3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutMma);
        *s_abort = 1;
      }
      umma_commit_pair(drain, 0x1);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, a.timeout_ns);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- epilogue (warps 2..5, both CTAs)
    // warp q reads TMEM lanes 32 q .. 32 q + 31: CTA rank's weight rows 32 q + lane of the item's tile
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool cleared = !(FUSED && EPI2 == kEpiCombineF32 && P.args[0].zero_out != nullptr);
    Seq sq;
    for (int p = seq_first(sq, lane == 0); __all_sync(0xffffffffu, sq.ok) && p >= 0;
         p = seq_next(sq, p, lane == 0)) {
      int ph, row0, nreal, n;
      WmCoord c;
      item(p, ph, c, row0, nreal, n);
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      if (ok && FUSED && ph == 1 && !cleared) {
        // the output this epilogue adds into: every clearing warp of the grid is done
        ok = wm_wait_count(&sched->wm_cleared, static_cast<uint32_t>(kZeroWarps * gridDim.x), s_abort, a.timeout_ns);
        cleared = true;
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * 256);
      if (ph == 0) {
        wm_epilogue<EPI>(P.args[0], c, row0, nreal, n, tbase, q, lane, static_cast<int>(rank), s_stage);
        if (FUSED) {
          // this warp's H stores: visible to the async proxy (TMA reads), then released to expert e's count
          wm_fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) wm_red_release_add(&sched->wm_done[c.e], 1u);
        }
      } else {
        if constexpr (FUSED)
          wm_epilogue<(EPI2 >= 0 ? EPI2 : EPI)>(P.args[1], c, row0, nreal, n, tbase, q, lane, static_cast<int>(rank),
                                               s_stage);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(tempty0 + 8 * acc);
        else
          mbar_arrive_peer(mapa_shared(tempty0 + 8 * acc, 0));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (a.zero_out != nullptr) {
    // -------------------------------------------------------------- clearing warps (up GEMM)
    clear_share(a.zero_out, a.zero_vec4, blockIdx.x, gridDim.x, threadIdx.x - 32 * kZeroWarp0);
    if (FUSED) {
      __syncwarp();
      if (lane == 0) wm_red_release_add(&sched->wm_cleared, 1u);
    }
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, WTMEM_COLS);
  }
}

template <int EPI, int EPI2>
cudaError_t launch_wm_t(const WmFused& f, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(f.args[0].zero_out ? WNUM_THREADS_ZERO : WNUM_THREADS);
  cfg.dynamicSmemBytes = WSMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_wm_gemm_kernel<EPI, EPI2>, f);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int EPI, int EPI2>
cudaError_t set_wm_smem() {
  return cudaFuncSetAttribute(tc_wm_gemm_kernel<EPI, EPI2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              WSMEM_BYTES);
}

}  // namespace

cudaError_t prepare_wm_gemm() {
  cudaError_t e = set_wm_smem<kEpiSwiGLU, -1>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiReluBias, -1>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiStoreF32, -1>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiCombineF32, -1>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiSwiGLU, kEpiCombineF32>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiSwiGLU, kEpiStoreF32>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiReluBias, kEpiCombineF32>();
  if (e == cudaSuccess) e = set_wm_smem<kEpiReluBias, kEpiStoreF32>();
  return e;
}

// Most CTAs of the weight-major kernel (pairs) resident at once on the current device (0 on error).
int wm_gemm_max_ctas() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(WNUM_THREADS_ZERO);
  cfg.dynamicSmemBytes = WSMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tc_wm_gemm_kernel<kEpiSwiGLU, kEpiCombineF32>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return 2 * clusters;
}

static bool wm_args_ok(const GemmArgs& a) {
  return a.wm_ntok >= 32 && a.wm_ntok <= 256 && (a.wm_ntok & 31) == 0 && a.n_per_expert % (2 * WBM) == 0 &&
         a.K > 0;
}

// grid: an even number of CTAs.  a.wm_ntok: token tile rows, a multiple of 32 in [32, 256].
cudaError_t launch_wm_gemm(int epi, const WmMaps& maps, const GemmArgs& a, int grid, cudaStream_t s) {
  grid &= ~1;
  if (grid <= 0) return cudaSuccess;
  if (!wm_args_ok(a)) return cudaErrorInvalidValue;
  WmFused f;
  f.maps[0] = maps;
  f.args[0] = a;
  f.maps[1] = maps;
  f.args[1] = a;
  switch (epi) {
    case kEpiSwiGLU:
      return launch_wm_t<kEpiSwiGLU, -1>(f, grid, s);
    case kEpiReluBias:
      return launch_wm_t<kEpiReluBias, -1>(f, grid, s);
    case kEpiCombineF32:
      return launch_wm_t<kEpiCombineF32, -1>(f, grid, s);
    default:
      return launch_wm_t<kEpiStoreF32, -1>(f, grid, s);
  }
}

// Both projections in one launch.  f.args[0]: the up projection (its tile_ctr is the one counter of
// the launch, its zero_out the output the down projection adds into); f.args[1]: the down projection
// (the same token tile, sched and E).  The counters wm_done / wm_cleared of f.args[0].sched must be
// zero (the router clears them).
cudaError_t launch_wm_fused(int epi_up, int epi_dn, const WmFused& f, int grid, cudaStream_t s) {
  grid &= ~1;
  if (grid <= 0) return cudaSuccess;
  if (!wm_args_ok(f.args[0]) || !wm_args_ok(f.args[1]) || f.args[0].wm_ntok != f.args[1].wm_ntok ||
      f.args[0].tile_ctr == nullptr)
    return cudaErrorInvalidValue;
  const bool swiglu = epi_up == kEpiSwiGLU;
  if (epi_up != kEpiSwiGLU && epi_up != kEpiReluBias) return cudaErrorInvalidValue;
  if (epi_dn == kEpiCombineF32)
    return swiglu ? launch_wm_t<kEpiSwiGLU, kEpiCombineF32>(f, grid, s) : launch_wm_t<kEpiReluBias, kEpiCombineF32>(f, grid, s);
  if (epi_dn == kEpiStoreF32)
    return swiglu ? launch_wm_t<kEpiSwiGLU, kEpiStoreF32>(f, grid, s) : launch_wm_t<kEpiReluBias, kEpiStoreF32>(f, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace colibri
