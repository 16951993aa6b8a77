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
constexpr int WSMEM_BYTES =
    1024 + WRING_BYTES + WSTG_BYTES + WNUM_BARS * 8 + 16 + 4 * (4 * kMaxE + 4 + WTQ);
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
__global__ void __launch_bounds__(WNUM_THREADS_ZERO, 1)
    tc_wm_gemm_kernel(const __grid_constant__ WmMaps maps, const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NT = a.wm_ntok;                           // token tile (multiple of 32, <= 256)
  const int stage_bytes = WA_BYTES + 64 * NT;         // weights + NT / 2 token rows of 128 bytes
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
  int* s_istart = s_tt + kMaxE + 1;
  volatile int* s_item = s_istart + kMaxE + 1;  // item-id queue

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + WSTAGES_MAX);
  const uint32_t tfull0 = smem_u32(bars + 2 * WSTAGES_MAX);
  const uint32_t tempty0 = smem_u32(bars + 2 * WSTAGES_MAX + 2);
  const uint32_t drain = smem_u32(bars + 2 * WSTAGES_MAX + 4);
  const uint32_t tqf0 = smem_u32(bars + 2 * WSTAGES_MAX + 5);
  const uint32_t tqe0 = smem_u32(bars + 2 * WSTAGES_MAX + 5 + WTQ);
  const bool DYN = a.tile_ctr != nullptr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int n_w = a.n_per_expert / (2 * WBM);  // 256-row weight tiles per expert

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
    prefetch_tmap(&maps.w);
    for (int i = 0; i < kWmTokMaps; ++i) prefetch_tmap(&maps.tok[i]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), WTMEM_COLS);
    tmem_relinquish_pair();
  }
  pdl_wait();  // the routing summary and the token rows come from earlier kernels
  if (a.clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.clear_word = 0u;
  if (threadIdx.x < kMaxE) s_counts[threadIdx.x] = threadIdx.x < E ? a.sched->counts[threadIdx.x] : 0;
  if (threadIdx.x < kMaxE + 1) s_offsets[threadIdx.x] = threadIdx.x <= E ? a.sched->offsets[threadIdx.x] : 0;
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_tt[e] = (s_counts[e] + NT - 1) / NT;
      s_istart[e] = acc;
      acc += n_w * s_tt[e];
    }
    s_istart[E] = acc;
  }
  tc_fence_before();
  cluster_sync();  // barrier inits and TMEM addresses visible across the pair
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = s_istart[E];
  const int num_kb = (a.K + WBK - 1) / WBK;
  const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  // the token tile of item c: first row, real rows, MMA width N (rows rounded up to 32)
  auto tile_rows = [&](const WmCoord& c, int& row0, int& nreal, int& n) {
    row0 = s_offsets[c.e] + c.t * NT;
    nreal = min(NT, s_counts[c.e] - c.t * NT);
    n = (nreal + 31) & ~31;
  };

  // Item order: pair i starts with item i; then (DYN) the leader's producer takes the next index
  // from a counter shared by all pairs and hands it to the pair's other roles through a WTQ-deep
  // queue in both CTAs' shared memory, else pair i takes items i, i + n_pairs, ...
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
  auto seq_first = [&]() -> int { return pair_id < total ? pair_id : -1; };
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
        const int p = n_pairs + static_cast<int>(atomicAdd(a.tile_ctr, 1u));
        return p < total ? p : -1;
      };
      int p = seq_first(), p_next = -1;
      for (; ok && p >= 0;) {
        const WmCoord c = decode_wm(p, s_istart, s_tt, E);
        int row0, nreal, n;
        tile_rows(c, row0, nreal, n);
        const int half_n = n / 2;
        const CUtensorMap* tm_tok = &maps.tok[half_n / 16 - 1];
        const int tok_row = row0 + static_cast<int>(rank) * half_n;
        const int wrow = c.e * a.n_per_expert + c.w * 2 * WBM;
        const uint32_t stage_tx = 2u * static_cast<uint32_t>(WA_BYTES + 128 * half_n);
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
          if constexpr (EPI == kEpiSwiGLU) {
            // gate rows 256 w + 64 rank + [0, 64) and their up rows 128 further on
            tma_load_2d_pair(sa, &maps.w, full_leader, kb * WBK, wrow + 64 * static_cast<int>(rank));
            tma_load_2d_pair(sa + WA_BYTES / 2, &maps.w, full_leader, kb * WBK, wrow + WBM + 64 * static_cast<int>(rank));
          } else {
            tma_load_2d_pair(sa, &maps.w, full_leader, kb * WBK, wrow + WBM * static_cast<int>(rank));
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
      int p = seq_first();
      bool ok = true;
      for (; ok && p >= 0; p = seq_next(sq, p, true), ok = ok && sq.ok) {
        int row0, nreal, n;
        tile_rows(decode_wm(p, s_istart, s_tt, E), row0, nreal, n);
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
    Seq sq;
    uint32_t* stg = s_stage + q * (32 * WSTG_LD);
    for (int p = seq_first(); __all_sync(0xffffffffu, sq.ok) && p >= 0; p = seq_next(sq, p, lane == 0)) {
      const WmCoord c = decode_wm(p, s_istart, s_tt, E);
      int row0, nreal, n;
      tile_rows(c, row0, nreal, n);
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * 256);
      const int nch = n / 32;
      if constexpr (EPI == kEpiSwiGLU) {
        // warps 0, 1: gate values of hidden units 64 rank + 32 q + lane; warps 2, 3: their up values
        const int f0 = c.w * WBM + 64 * static_cast<int>(rank) + 32 * (q & 1);  // this warp pair's units
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
              const int idx = 32 * i + lane, j = idx >> 2, g8 = idx & 3;  // token j, 8 units 8 g8..
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
        const int f0 = c.w * 2 * WBM + WBM * static_cast<int>(rank) + 32 * q;  // this warp's 32 units
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
        const int d0 = c.w * 2 * WBM + WBM * static_cast<int>(rank) + 32 * q;
        const float b = a.bias ? a.bias[static_cast<size_t>(c.e) * a.out_cols + d0 + lane] : 0.f;
#pragma unroll 1
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          // token and gate (or output row) of the chunk's token lane
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
            const int idx = 32 * i + lane, j = idx >> 3, g4 = idx & 7;  // token j, columns 4 g4..
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
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, WTMEM_COLS);
  }
}

template <int EPI>
cudaError_t launch_wm_t(const WmMaps& maps, const GemmArgs& a, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(a.zero_out ? WNUM_THREADS_ZERO : WNUM_THREADS);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_wm_gemm_kernel<EPI>, maps, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t prepare_wm_gemm() {
  cudaError_t e = cudaSuccess;
  for (auto k : {tc_wm_gemm_kernel<kEpiSwiGLU>, tc_wm_gemm_kernel<kEpiReluBias>, tc_wm_gemm_kernel<kEpiStoreF32>,
                 tc_wm_gemm_kernel<kEpiCombineF32>})
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, WSMEM_BYTES);
  return e;
}

// grid: an even number of CTAs, at most the co-resident pairs of the CTA-pair kernel (same shared
// memory footprint class).  a.wm_ntok: token tile rows, a multiple of 32 in [32, 256].
cudaError_t launch_wm_gemm(int epi, const WmMaps& maps, const GemmArgs& a, int grid, cudaStream_t s) {
  grid &= ~1;
  if (grid <= 0) return cudaSuccess;
  if (a.wm_ntok < 32 || a.wm_ntok > 256 || (a.wm_ntok & 31) || (a.n_per_expert % (2 * WBM))) return cudaErrorInvalidValue;
  switch (epi) {
    case kEpiSwiGLU:
      return launch_wm_t<kEpiSwiGLU>(maps, a, grid, s);
    case kEpiReluBias:
      return launch_wm_t<kEpiReluBias>(maps, a, grid, s);
    case kEpiCombineF32:
      return launch_wm_t<kEpiCombineF32>(maps, a, grid, s);
    default:
      return launch_wm_t<kEpiStoreF32>(maps, a, grid, s);
  }
}

}  // namespace colibri
