// Grouped expert GEMM on CTA pairs (tcgen05 cta_group::2): 256x256 output tiles.
//
// Same computation as gemm_tcgen05.cu (the Compute stage of zskr.cn/news/2272131, "Colibri: a
// lightweight C MoE inference engine for edge devices", 2.1: one GEMM per expert over its
// contiguous rows, activation fused in the epilogue as in m.nxbn.cn/news/48047 2.1), mapped onto a
// cluster of two CTAs on neighbouring SMs:
//
//   - each CTA loads its own 128-row A tile (its own M rows) and one 128-row half of the 256-row B
//     tile, so each SM stages 32 KB per 64-wide K step instead of 48 KB;
//   - the leader CTA (rank 0) issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16), which reads A and
//     B from both CTAs' shared memory and accumulates each CTA's 128 rows in that CTA's TMEM;
//   - both CTAs' TMA loads complete on the leader's `full` barrier; the leader's commits multicast to
//     both CTAs' `empty` and `tmem_full` barriers; both epilogues arrive on the leader's `tmem_empty`.
//
// A pair computes two 128-row M tiles of one expert that share the weight tile; when an expert has
// an odd number of M tiles, the second CTA of its last pair computes rows past the expert's segment
// (read as they are or as zeros past the buffer) and stores nothing.  Waits are bounded as in the
// single-CTA kernel; TMEM is allocated and freed collectively by one warp of each CTA.  Tiles are
// handed out in index order at run time (see "Tile order" below).  The up projection can carry two
// more warps that clear the fused combine's output while the mainloop runs.
//
// Gathered A (GA, up projection): the A rows come straight from the token rows x through
// token_of_row (gather_a.cuh); extra warps of each CTA copy them with cp.async and a forwarder
// thread of each CTA arrives on the leader's `full` barrier once they are in place, next to the
// TMA bytes of B.  The MMA issuer waits on `full` with a cluster-scope acquire.
#include "gather_a.cuh"

namespace colibri {
namespace {

using namespace ptx;

constexpr int PBM = 128, PBN = 256, PBK = 64, PUMMA_K = 16;
constexpr int PSTAGES = 6;
constexpr int PA_BYTES = PBM * PBK * 2;         // 16 KB: this CTA's A rows
constexpr int PB_BYTES = (PBN / 2) * PBK * 2;   // 16 KB: this CTA's half of B
constexpr int PSTAGE_BYTES = PA_BYTES + PB_BYTES;
constexpr int PNUM_THREADS = 192;
constexpr int PNUM_THREADS_ZERO = 192 + 32 * kZeroWarps;  // + the warps clearing out (up GEMM)
constexpr int PNUM_THREADS_GA = 192 + 32 * (kGatherWarps + kForwarders);  // + A gather and forwarder warps
constexpr uint32_t PTMEM_COLS = 512;
constexpr int PTQ = 4;  // tile-id queue depth (dynamic tile order)
constexpr int kPublishAt = 4;  // stage of a tile at which the leader hands out the next tile's index
// full, empty, tmem_full[2], tmem_empty[2], drain, gfull, tile queue full / empty
constexpr int PNUM_BARS = 3 * PSTAGES + 5 + 2 * PTQ;
// Epilogue staging: each epilogue warp turns its 32 rows x 32 words of a chunk around in shared
// memory (row stride 36 words: both the row-per-thread writes and the 4-rows-per-instruction reads
// are free of bank conflicts), so that every global write instruction covers four whole 128-byte row
// segments instead of 16 bytes of 32 different rows.
constexpr int PSTG_LD = 36;
constexpr int PSTG_BYTES = 4 * 32 * PSTG_LD * 4;  // 4 warps x 32 rows x 36 words
constexpr int PSMEM_BYTES =
    1024 + PSTAGES * PSTAGE_BYTES + PSTG_BYTES + PNUM_BARS * 8 + 16 + 4 * (4 * kMaxE + 4 + PTQ);
static_assert(PSMEM_BYTES <= 227 * 1024, "pair GEMM shared memory");
static_assert(PSTAGES % kForwarders == 0, "a stage keeps its forwarder across ring cycles");

struct PairCoord {
  int e, pm, n;
  bool half;  // the expert's odd last 128-row M tile alone: an M=128 pair tile (64 rows per CTA)
};

// Tile p -> (expert, pair of 128-row M tiles, N tile).  An expert with an odd number of M tiles
// ends with a pair whose second tile lies past its rows; with allow_half that pair is computed as
// one M=128 tile instead of an M=256 tile half of padding.
__device__ __forceinline__ PairCoord decode_pair(int p, const int* pstart, const int* mstart, int E, int n_tiles,
                                                 bool allow_half) {
  int e = 0;
  while (e + 1 < E && pstart[e + 1] * n_tiles <= p) ++e;
  const int local = p - pstart[e] * n_tiles;
  const int pme = pstart[e + 1] - pstart[e];
  PairCoord c;
  c.e = e;
  c.n = local / pme;
  c.pm = local - c.n * pme;
  c.half = allow_half && 2 * c.pm + 1 == mstart[e + 1] - mstart[e];
  return c;
}

// Epilogue warps q and q ^ 2 of a half tile hold the two column halves of the same 32 rows (see the
// M=128 TMEM layout in the kernel); they meet at named barrier 2 + (q & 1), 64 threads.
__device__ __forceinline__ void pair_warps_sync(int q) {
  if (q & 1)
    asm volatile("bar.sync 3, 64;" ::: "memory");
  else
    asm volatile("bar.sync 2, 64;" ::: "memory");
}

template <int EPI, bool GA>
__global__ void __launch_bounds__(GA ? PNUM_THREADS_GA : PNUM_THREADS_ZERO, 1)
    tc_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmA64, const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + PSTAGES * PA_BYTES;
  uint32_t* s_stage = reinterpret_cast<uint32_t*>(sB + PSTAGES * PB_BYTES);  // epilogue staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s_stage) + PSTG_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + PNUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_counts = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_offsets = s_counts + kMaxE;
  int* s_mstart = s_offsets + kMaxE + 1;
  int* s_pstart = s_mstart + kMaxE + 1;
  volatile int* s_tile = s_pstart + kMaxE + 1;  // tile-id queue (dynamic order)

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + PSTAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * PSTAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * PSTAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * PSTAGES + 4);
  const uint32_t gfull0 = smem_u32(bars + 2 * PSTAGES + 5);  // gathered A: rows of a stage landed
  const uint32_t tqf0 = smem_u32(bars + 3 * PSTAGES + 5);     // tile queue: slot written (each CTA)
  const uint32_t tqe0 = smem_u32(bars + 3 * PSTAGES + 5 + PTQ);  // tile queue: slot read (leader's)
  const bool DYN = !GA && a.tile_ctr != nullptr;  // tiles handed out in order at run time (see below)
  const bool HALF = !GA && a.half_tiles != 0;     // an expert's odd last M tile as an M=128 pair tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      // leader's: one arrive with both CTAs' TMA bytes per phase (+ each CTA's A forwarder)
      mbar_init(full0 + 8 * s, GA ? 3 : 1);
      mbar_init(empty0 + 8 * s, 1);  // each CTA's: one multicast commit per phase
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 8);  // leader's: 4 epilogue warps of each CTA
    }
    mbar_init(drain, 1);
    if constexpr (GA)
      for (int s = 0; s < PSTAGES; ++s) mbar_init(gfull0 + 8 * s, kGatherThreads);
    for (int i = 0; i < PTQ; ++i) {
      mbar_init(tqf0 + 8 * i, 1);   // the leader's producer
      mbar_init(tqe0 + 8 * i, 10);  // leader: MMA + 4 epilogue warps; peer: producer + 4 epilogue warps
    }
    *s_abort = 0;
    fence_mbar_init();
    if constexpr (!GA) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmA64);
    }
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), PTMEM_COLS);
    tmem_relinquish_pair();
  }
  pdl_wait();  // the routing summary and the A operand come from earlier kernels
  // the router (whose dispatch is fused) has completed: its grid barrier counter is free again
  if (a.clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.clear_word = 0u;
  if (threadIdx.x < kMaxE) s_counts[threadIdx.x] = threadIdx.x < E ? a.sched->counts[threadIdx.x] : 0;
  if (threadIdx.x < kMaxE + 1) {
    s_offsets[threadIdx.x] = threadIdx.x <= E ? a.sched->offsets[threadIdx.x] : 0;
    s_mstart[threadIdx.x] = threadIdx.x <= E ? a.sched->mtile_start[threadIdx.x] : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_pstart[e] = acc;
      acc += (s_mstart[e + 1] - s_mstart[e] + 1) / 2;
    }
    s_pstart[E] = acc;
  }
  tc_fence_before();
  cluster_sync();  // barrier inits and TMEM addresses visible across the pair
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = s_pstart[E] * a.n_tiles;
  const int num_kb = (a.K + PBK - 1) / PBK;
  const int pair_id = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;

  // Tile order.  Static: pair i takes tiles i, i + n_pairs, ...  Dynamic (DYN): pair i starts with
  // tile i; after that the leader's producer takes the next tile index from a counter shared by all
  // pairs (n_pairs + one atomic per tile, fetched while the current tile's first stage is in flight)
  // and hands it to the pair's other roles through a PTQ-deep queue in both CTAs' shared memory, so
  // tiles run in index order whatever the pairs' speeds: the pairs that share a weight tile
  // (consecutive indices) stay together and read it from L2, where a static order lets them drift
  // apart over a launch.
  struct Seq {
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
  };
  auto take = [&](Seq& sq, bool arrive) -> int {  // next id from this CTA's queue; -1 = no more
    if (!mbar_wait_cluster(tqf0 + 8 * sq.slot, sq.ph, s_abort, a.timeout_ns)) {
      sq.ok = false;
      return -1;
    }
    const int p = s_tile[sq.slot];
    if (arrive) {
      if (leader)
        mbar_arrive(tqe0 + 8 * sq.slot);
      else
        mbar_arrive_peer(mapa_shared(tqe0 + 8 * sq.slot, 0));
    }
    if (++sq.slot == PTQ) {
      sq.slot = 0;
      sq.ph ^= 1u;
    }
    return p;
  };
  auto seq_first = [&](Seq& sq, bool arrive) -> int {  // the first tile is pair_id in both orders
    (void)sq;
    (void)arrive;
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
      Seq sq, pub;  // pub: the leader's publishing position in the queue
      auto publish = [&](int p) -> bool {
        if (!mbar_wait(tqe0 + 8 * pub.slot, pub.ph ^ 1u, s_abort, a.timeout_ns)) return false;
        s_tile[pub.slot] = p;
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(s_tile + pub.slot)), 1), p);
        mbar_arrive(tqf0 + 8 * pub.slot);
        mbar_arrive_remote(mapa_shared(tqf0 + 8 * pub.slot, 1));  // release.cluster: the id is there
        if (++pub.slot == PTQ) {
          pub.slot = 0;
          pub.ph ^= 1u;
        }
        return true;
      };
      auto fetch = [&]() -> int {
        const int p = n_pairs + static_cast<int>(atomicAdd(a.tile_ctr, 1u));
        return p < total ? p : -1;
      };
      int p = seq_first(sq, true), p_next = -1;
      for (; ok && p >= 0;) {
        const PairCoord c = decode_pair(p, s_pstart, s_mstart, E, a.n_tiles, HALF);
        // full tile: this CTA's 128-row M tile; half tile: its 64 rows of the one M tile
        const int a_row = c.half ? s_offsets[c.e] + 2 * c.pm * PBM + static_cast<int>(rank) * (PBM / 2)
                                 : s_offsets[c.e] + (2 * c.pm + static_cast<int>(rank)) * PBM;
        const int b_row = c.e * a.n_per_expert + c.n * PBN + static_cast<int>(rank) * (PBN / 2);
        const uint32_t stage_tx = GA ? 2 * PB_BYTES : (c.half ? 2 * (PA_BYTES / 2 + PB_BYTES) : 2 * PSTAGE_BYTES);
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
          if constexpr (!GA)
            tma_load_2d_pair(smem_u32(sA + stage * PA_BYTES), c.half ? &tmA64 : &tmA, full_leader, kb * PBK, a_row);
          tma_load_2d_pair(smem_u32(sB + stage * PB_BYTES), &tmB, full_leader, kb * PBK, b_row);
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
          // the next tile: its index requested with this tile's first stage, handed to the pair a few
          // stages later (the atomic's latency and the cluster-scope release then overlap the copies)
          if (DYN && leader && kb == 0) p_next = fetch();
          if (DYN && leader && kb == (num_kb > kPublishAt ? kPublishAt : num_kb - 1)) {
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
      for (int s = 0; s < PSTAGES; ++s)
        if (armed & (1u << s)) {
          volatile int never = 0;
          mbar_wait(full0 + 8 * s, (armed_phase >> s) & 1u, &never, a.timeout_ns);
        }
    }
  } else if (GA && warp >= kGatherWarp0 && warp < kForwardWarp0) {
    // -------------------------------------------------------------- A gather warps
    AGather g;
    g.init(a.gather_x, a.K, warp - kGatherWarp0, lane);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    auto prefetch = [&](int p) {
      if (p >= total) return;
      const PairCoord c = decode_pair(p, s_pstart, s_mstart, E, a.n_tiles, false);
      g.prefetch_tokens(a.token_of_row, s_offsets[c.e] + (2 * c.pm + static_cast<int>(rank)) * PBM,
                        s_offsets[c.e] + s_counts[c.e]);
    };
    prefetch(pair_id);
    for (int p = pair_id; ok && p < total; p += n_pairs) {
      g.advance_tile();
      prefetch(p + n_pairs);
      for (int kb = 0; kb < num_kb; ++kb) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(empty0 + 8 * stage, phase ^ 1u, s_abort, a.timeout_ns));
        if (!got) {
          ok = false;
          break;
        }
        g.issue(smem_u32(sA + stage * PA_BYTES), kb);
        cp_async_arrive_noinc(gfull0 + 8 * stage);
        if (++stage == PSTAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait<0>();  // nothing of this thread in flight when the CTA leaves
    if (!ok && lane == 0) {
      if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
      *s_abort = 1;
    }
  } else if (GA && warp >= kForwardWarp0) {
    // -------------------------------------------------------------- A forwarders (lane 0 of each forwarder warp)
    // forwarder f handles the stages s with s % kForwarders == f, so the per-stage wake-up, proxy
    // fence and arrive of consecutive stages overlap
    const int fwd = warp - kForwardWarp0;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int p = pair_id; ok && p < total; p += n_pairs) {
        for (int kb = 0; kb < num_kb; ++kb) {
          if (stage % kForwarders == fwd) {
            if (!mbar_wait(gfull0 + 8 * stage, phase, s_abort, a.timeout_ns)) {
              ok = false;
              break;
            }
            fence_proxy_async_smem();
            mbar_arrive_peer(mapa_shared(full0 + 8 * stage, 0));
          }
          if (++stage == PSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
        *s_abort = 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ MMA issuer (leader only)
      constexpr uint32_t idesc_full = make_idesc_bf16(2 * PBM, PBN);
      constexpr uint32_t idesc_half = make_idesc_bf16(PBM, PBN);  // M=128: 64 rows from each CTA
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      Seq sq;
      int p = seq_first(sq, true);
      bool ok = sq.ok;
      for (; ok && p >= 0; p = seq_next(sq, p, true), ok = ok && sq.ok) {
        if (!mbar_wait_cluster(tempty0 + 8 * acc, acc_phase ^ 1u, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t idesc = decode_pair(p, s_pstart, s_mstart, E, a.n_tiles, HALF).half ? idesc_half : idesc_full;
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PBN);
        for (int kb = 0; kb < num_kb; ++kb) {
          const bool got = GA ? mbar_wait_cluster(full0 + 8 * stage, phase, s_abort, a.timeout_ns)
                              : mbar_wait(full0 + 8 * stage, phase, s_abort, a.timeout_ns);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * PA_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * PB_BYTES);
#pragma unroll
          for (int k = 0; k < PBK / PUMMA_K; ++k)
            umma_bf16_pair(d_tmem, sw128_desc(a_addr + k * PUMMA_K * 2), sw128_desc(b_addr + k * PUMMA_K * 2), idesc,
                           (kb | k) != 0 ? 1u : 0u);
          umma_commit_pair(empty0 + 8 * stage, 0x3);
          if (++stage == PSTAGES) {
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
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    Seq sq;
    for (int p = seq_first(sq, lane == 0); __all_sync(0xffffffffu, sq.ok) && p >= 0; p = seq_next(sq, p, lane == 0)) {
      const PairCoord c = decode_pair(p, s_pstart, s_mstart, E, a.n_tiles, HALF);
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      // this warp's rows.  Full tile (M=256): TMEM lane l of this CTA = row l of its 128-row M tile.
      // Half tile (M=128, measured on GB300): this CTA's 64 rows sit in lanes 0..63 with output
      // columns 0..127 of the tile and again in lanes 64..127 with columns 128..255, both in
      // accumulator columns 0..127 -- so warp q holds rows 32 * (q & 1) + lane, column half q >> 1.
      const int row0 = c.half ? s_offsets[c.e] + 2 * c.pm * PBM + static_cast<int>(rank) * (PBM / 2) + (q & 1) * 32
                              : s_offsets[c.e] + (2 * c.pm + static_cast<int>(rank)) * PBM + q * 32;
      const int nch = c.half ? 4 : PBN / 32;          // 32-column accumulator chunks this warp drains
      const int coff = c.half ? (q >> 1) * 128 : 0;   // first output column of the tile those hold
      const int seg_end = s_offsets[c.e] + s_counts[c.e];
      const bool valid = row0 + lane < seg_end;  // this thread's row (the TMEM lane it reads)
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * PBN);
      // write-back mapping: lane -> row 4 * i + rr of the warp's 32 (i = 0..7), 16-byte column group cg
      const int rr = lane >> 3, cg = lane & 7;
      uint32_t* stg = s_stage + q * (32 * PSTG_LD);
      uint32_t* stg_mine = stg + lane * PSTG_LD;          // row-per-thread side
      const uint32_t* stg_wb = stg + rr * PSTG_LD + 4 * cg;  // + 4 * i * PSTG_LD: write-back side
      // rows of the write-back side that exist: bit i for row 4 * i + rr
      uint32_t wb_valid = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) wb_valid |= (row0 + 4 * i + rr < seg_end ? 1u : 0u) << i;
      // a chunk pair of bf16 results (64 columns, 128 bytes per row) from the staging tile to rows of `out`
      auto write_bf16_rows = [&](__nv_bfloat16* out, int64_t ldo) {
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 val = *reinterpret_cast<const uint4*>(stg_wb + 4 * i * PSTG_LD);
          if ((wb_valid >> i) & 1u)
            *reinterpret_cast<uint4*>(out + static_cast<size_t>(row0 + 4 * i + rr) * ldo + 8 * cg) = val;
        }
        __syncwarp();  // the staging tile is rewritten next
      };
      if constexpr (EPI == kEpiSwiGLU) {
        // columns [0,128) = gate (B half of the leader), [128,256) = up (B half of the peer)
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + c.n * (PBN / 2);
        if (c.half) {
          // half tile: the gate values of rows 32 * (q & 1) + lane are with warp q < 2, their up values
          // with warp q + 2, which hands each 32-column chunk over through its own staging tile
          const uint4* stg_up = reinterpret_cast<const uint4*>(s_stage + (q ^ 2) * (32 * PSTG_LD) + lane * PSTG_LD);
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld32_sync(tbase + ch * 32, v);
            if (q >= 2) {
              uint4* dst = reinterpret_cast<uint4*>(stg_mine);
#pragma unroll
              for (int w = 0; w < 8; ++w) dst[w] = make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
              pair_warps_sync(q);  // up values in place
              pair_warps_sync(q);  // taken by the gate warp
            } else {
              uint32_t u[32];
              pair_warps_sync(q);
#pragma unroll
              for (int w = 0; w < 8; ++w) {
                const uint4 t = stg_up[w];
                u[4 * w] = t.x;
                u[4 * w + 1] = t.y;
                u[4 * w + 2] = t.z;
                u[4 * w + 3] = t.w;
              }
              pair_warps_sync(q);
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float g0 = __uint_as_float(v[2 * i]), g1 = __uint_as_float(v[2 * i + 1]);
                const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                pk[i] = pack_bf16(silu_fast(g0) * u0, silu_fast(g1) * u1);
              }
              uint4* dst = reinterpret_cast<uint4*>(stg_mine + 16 * (ch & 1));
#pragma unroll
              for (int w = 0; w < 4; ++w) dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
              if (ch & 1) write_bf16_rows(out + (ch - 1) * 32, a.ldo);
            }
          }
        } else
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t g[32], u[32];
          tmem_ld32_sync(tbase + ch * 32, g);
          tmem_ld32_sync(tbase + 128 + ch * 32, u);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            pk[i] = pack_bf16(silu_fast(g0) * u0, silu_fast(g1) * u1);
          }
          uint4* dst = reinterpret_cast<uint4*>(stg_mine + 16 * (ch & 1));
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          if (ch & 1) write_bf16_rows(out + (ch - 1) * 32, a.ldo);
        }
      } else if constexpr (EPI == kEpiReluBias) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + c.n * PBN + coff;
        const float* bias = a.bias + static_cast<size_t>(c.e) * a.out_cols + c.n * PBN + coff;
#pragma unroll 1
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16(fmaxf(__uint_as_float(v[2 * i]) + bias[ch * 32 + 2 * i], 0.f),
                              fmaxf(__uint_as_float(v[2 * i + 1]) + bias[ch * 32 + 2 * i + 1], 0.f));
          uint4* dst = reinterpret_cast<uint4*>(stg_mine + 16 * (ch & 1));
#pragma unroll
          for (int w = 0; w < 4; ++w) dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
          if (ch & 1) write_bf16_rows(out + (ch - 1) * 32, a.ldo);
        }
      } else {
        // fp32 results: Y rows, or (kEpiCombineF32) out[token] += gate * (acc (+ b2)); with two slots
        // and a zeroed output the two reductions give RN(g0*y0 + g1*y1) in either order, the value the
        // separate combine computes
        constexpr bool kCombine = EPI == kEpiCombineF32;
        const float* bias = a.bias ? a.bias + static_cast<size_t>(c.e) * a.out_cols + c.n * PBN : nullptr;
        // token and gate of the write-back side's rows (those of row 4 * i + rr sit in lane 4 * i + rr)
        // (kEpiStoreF32 with a row map: the output row of each A row, e.g. receive order on an expert rank)
        const int my_tok = kCombine && valid ? __ldcg(a.token_of_row + row0 + lane)
                           : (!kCombine && a.row_map != nullptr && valid ? __ldcg(a.row_map + row0 + lane) : 0);
        const float my_g = kCombine && valid ? __ldcg(a.gate_of_row + row0 + lane) : 0.f;
        int tok[8];
        float gr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          tok[i] = __shfl_sync(0xffffffffu, my_tok, 4 * i + rr);
          gr[i] = __shfl_sync(0xffffffffu, my_g, 4 * i + rr);
        }
#pragma unroll 1
        for (int ch = 0; ch < nch; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          uint4* dst = reinterpret_cast<uint4*>(stg_mine);
#pragma unroll
          for (int w = 0; w < 8; ++w) dst[w] = make_uint4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
          __syncwarp();
          const int col = coff + ch * 32 + 4 * cg;  // this lane's 4 columns of the chunk
          float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (bias) b4 = make_float4(bias[col], bias[col + 1], bias[col + 2], bias[col + 3]);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 raw = *reinterpret_cast<const uint4*>(stg_wb + 4 * i * PSTG_LD);
            float y[4] = {__uint_as_float(raw.x), __uint_as_float(raw.y), __uint_as_float(raw.z),
                          __uint_as_float(raw.w)};
            if (bias) {
              y[0] += b4.x;
              y[1] += b4.y;
              y[2] += b4.z;
              y[3] += b4.w;
            }
            if ((wb_valid >> i) & 1u) {
              if constexpr (kCombine) {
                float* o = static_cast<float*>(a.out) + static_cast<size_t>(tok[i]) * a.ldo + c.n * PBN + col;
                red_add_v4(o, __fmul_rn(gr[i], y[0]), __fmul_rn(gr[i], y[1]), __fmul_rn(gr[i], y[2]),
                           __fmul_rn(gr[i], y[3]));
              } else {
                const int orow = a.row_map != nullptr ? tok[i] : row0 + 4 * i + rr;
                float* o = static_cast<float*>(a.out) + static_cast<size_t>(orow) * a.ldo + c.n * PBN + col;
                *reinterpret_cast<float4*>(o) = make_float4(y[0], y[1], y[2], y[3]);
              }
            }
          }
          __syncwarp();  // the staging tile is rewritten next
        }
      }
      tc_fence_before();
      __syncwarp();
      // accumulator free: the leader's barrier; the peer arrives with the default CTA-scope release
      // (a cluster-scope release costs about a microsecond per arrival; nothing but the tcgen05 loads
      // fenced above is ordered by it) and the MMA issuer acquires at cluster scope
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
  } else if (!GA && a.zero_out != nullptr) {
    // -------------------------------------------------------------- clearing warps (up GEMM)
    clear_share(a.zero_out, a.zero_vec4, blockIdx.x, gridDim.x, threadIdx.x - 32 * kZeroWarp0);
  }

  tc_fence_before();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, PTMEM_COLS);
  }
}

template <int EPI, bool GA>
cudaError_t launch_pair_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmA64, const GemmArgs& a,
                          int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(GA ? PNUM_THREADS_GA : (a.zero_out ? PNUM_THREADS_ZERO : PNUM_THREADS));
  cfg.dynamicSmemBytes = PSMEM_BYTES;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, tc_pair_gemm_kernel<EPI, GA>, tmA, tmB, tmA64, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

template <int EPI, bool GA>
cudaError_t set_pair_smem() {
  return cudaFuncSetAttribute(tc_pair_gemm_kernel<EPI, GA>, cudaFuncAttributeMaxDynamicSharedMemorySize, PSMEM_BYTES);
}

cudaError_t prepare_pair_gemm() {
  cudaError_t e = set_pair_smem<kEpiSwiGLU, false>();
  if (e == cudaSuccess) e = set_pair_smem<kEpiSwiGLU, true>();
  if (e == cudaSuccess) e = set_pair_smem<kEpiReluBias, false>();
  if (e == cudaSuccess) e = set_pair_smem<kEpiReluBias, true>();
  if (e == cudaSuccess) e = set_pair_smem<kEpiStoreF32, false>();
  if (e == cudaSuccess) e = set_pair_smem<kEpiCombineF32, false>();
  return e;
}

// Most CTA pairs of this kernel that can be resident at once on the current device (0 on error).
int pair_gemm_max_ctas() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PNUM_THREADS);
  cfg.dynamicSmemBytes = PSMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tc_pair_gemm_kernel<kEpiStoreF32, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return 2 * clusters;
}

// grid: an even number of CTAs (one pair per two SMs).  tmA64: the A operand with 64-row boxes (an
// expert's odd last M tile runs as an M=128 pair tile).  gather_a: A rows are gathered from
// a.gather_x through a.token_of_row (up-projection epilogues only) and tmA / tmA64 are not read.
cudaError_t launch_pair_gemm(int epi, bool gather_a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                             const CUtensorMap& tmB, const GemmArgs& a, int grid, cudaStream_t s) {
  grid &= ~1;
  if (grid <= 0) return cudaSuccess;
  switch (epi) {
    case kEpiSwiGLU:
      return gather_a ? launch_pair_t<kEpiSwiGLU, true>(tmA, tmB, tmA64, a, grid, s)
                      : launch_pair_t<kEpiSwiGLU, false>(tmA, tmB, tmA64, a, grid, s);
    case kEpiReluBias:
      return gather_a ? launch_pair_t<kEpiReluBias, true>(tmA, tmB, tmA64, a, grid, s)
                      : launch_pair_t<kEpiReluBias, false>(tmA, tmB, tmA64, a, grid, s);
    case kEpiCombineF32:
      if (gather_a) return cudaErrorInvalidValue;
      return launch_pair_t<kEpiCombineF32, false>(tmA, tmB, tmA64, a, grid, s);
    default:
      if (gather_a) return cudaErrorInvalidValue;
      return launch_pair_t<kEpiStoreF32, false>(tmA, tmB, tmA64, a, grid, s);
  }
}

}  // namespace colibri
