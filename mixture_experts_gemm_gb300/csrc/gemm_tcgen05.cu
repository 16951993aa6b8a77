// Grouped expert GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), operands by TMA.
//
// The Compute stage of zskr.cn/news/2272131 ("Colibri: a lightweight C MoE inference engine for
// edge devices") 2.1 is a grouped GEMM, one GEMM per expert over that expert's contiguous rows;
// the expert weights sit in one contiguous block per expert (2.2), each expert is an affine map
// with W stored [out, in] (hnwysp.cn/news/30485 3.2), and the activation is fused into the expert
// kernel (m.nxbn.cn/news/48047 2.1).  Here:
//
//   C[rows_e, n-tile] = A[rows_e, K] * B_e[n-tile, K]^T       bf16 x bf16 -> fp32 in TMEM
//
// A = expert-contiguous activations (Xp for the up projection, H for the down projection), both
// operands K-major, which is the nn.Linear [out, in] layout as stored.
//
// Design (one CTA per SM, persistent, warp-specialised, 192 threads):
//   warp 0      TMA producer: 128x64 A tile + 256x64 B tile per stage, 128-byte swizzle,
//               STAGES-deep shared-memory ring guarded by full/empty mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators), one lane issues
//               tcgen05.mma (M=128, N=256, K=16, kind::f16 with bf16 inputs) and commits each
//               stage back to the producer and each finished accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time, activation, store.  The two
//               accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// Tiles are (expert, 128-row tile, 256-column tile), row tile fastest, so CTAs that run at the same
// time share one weight tile (read once from HBM, then from L2) while the expert's activation rows
// stay L2-resident.  Expert segments are padded to 128 rows, so a tile never spans two experts;
// rows past the expert's count are computed but not stored.
//
// Every mbarrier wait is bounded (GemmArgs::timeout_ns): on expiry the kernel raises a bit in the
// device status word, stops all roles, waits (bounded) for its own TMA copies and MMAs, frees
// TMEM and returns.
//
// Gathered A (GA, up projection only): A rows come straight from the token rows x through
// token_of_row (gather_a.cuh): extra warps copy them with cp.async, and a forwarder thread arrives
// on `full` once they are in place, next to the TMA bytes of B.
#include "gather_a.cuh"

namespace colibri {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64, UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int NUM_THREADS_ZERO = 192 + 32 * kZeroWarps;  // + the warps clearing out (up GEMM)
constexpr int NUM_THREADS_GA = 192 + 32 * (kGatherWarps + kForwarders);  // + A gather and forwarder warps
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_BARS = 3 * STAGES + 5;  // full, empty, tmem_full[2], tmem_empty[2], drain, gfull
static_assert(STAGES % kForwarders == 0, "a stage keeps its forwarder across ring cycles");
constexpr int SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 + 4 * (3 * kMaxE + 3);

struct TileCoord {
  int e, m, n;
};

// tile -> (expert, row tile inside the expert, column tile); row tiles fastest.
__device__ __forceinline__ TileCoord decode_tile(int tile, const int* mtile_start, int E, int n_tiles) {
  int e = 0;
  while (e + 1 < E && mtile_start[e + 1] * n_tiles <= tile) ++e;
  const int local = tile - mtile_start[e] * n_tiles;
  const int mt = mtile_start[e + 1] - mtile_start[e];
  TileCoord c;
  c.e = e;
  c.n = local / mt;
  c.m = local - c.n * mt;
  return c;
}

template <int EPI, bool GA>
__global__ void __launch_bounds__(GA ? NUM_THREADS_GA : NUM_THREADS_ZERO, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_counts = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_offsets = s_counts + kMaxE;
  int* s_mstart = s_offsets + kMaxE + 1;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t gfull0 = smem_u32(bars + 2 * STAGES + 5);  // gathered A: rows of a stage landed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, GA ? 2 : 1);  // TMA arrive (+ the A forwarder)
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 4);
    }
    mbar_init(drain, 1);
    if constexpr (GA)
      for (int s = 0; s < STAGES; ++s) mbar_init(gfull0 + 8 * s, kGatherThreads);
    *s_abort = 0;
    fence_mbar_init();
    if constexpr (!GA) prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  pdl_wait();  // the routing summary and the A operand come from earlier kernels
  // the router (whose dispatch is fused) has completed: its grid barrier counter is free again
  if (a.clear_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.clear_word = 0u;
  if (threadIdx.x < kMaxE) s_counts[threadIdx.x] = threadIdx.x < E ? a.sched->counts[threadIdx.x] : 0;
  if (threadIdx.x < kMaxE + 1) {
    s_offsets[threadIdx.x] = threadIdx.x <= E ? a.sched->offsets[threadIdx.x] : 0;
    s_mstart[threadIdx.x] = threadIdx.x <= E ? a.sched->mtile_start[threadIdx.x] : 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total_tiles = s_mstart[E] * a.n_tiles;
  const int num_kb = (a.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: full[s] armed at least once
      uint32_t armed_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, s_mstart, E, a.n_tiles);
        const int a_row = s_offsets[c.e] + c.m * BM;
        const int b_row = c.e * a.n_per_expert + c.n * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full0 + 8 * stage, GA ? B_BYTES : STAGE_BYTES);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if constexpr (!GA) tma_load_2d(smem_u32(sA + stage * A_BYTES), &tmA, full0 + 8 * stage, kb * BK, a_row);
          tma_load_2d(smem_u32(sB + stage * B_BYTES), &tmB, full0 + 8 * stage, kb * BK, b_row);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
        *s_abort = 1;
      }
      // wait (bounded) for every copy this thread issued to land before the CTA can exit
      for (int s = 0; s < STAGES; ++s)
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
    auto prefetch = [&](int tile) {
      if (tile >= total_tiles) return;
      const TileCoord c = decode_tile(tile, s_mstart, E, a.n_tiles);
      g.prefetch_tokens(a.token_of_row, s_offsets[c.e] + c.m * BM, s_offsets[c.e] + s_counts[c.e]);
    };
    prefetch(blockIdx.x);
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      g.advance_tile();
      prefetch(tile + gridDim.x);
      for (int kb = 0; kb < num_kb; ++kb) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(empty0 + 8 * stage, phase ^ 1u, s_abort, a.timeout_ns));
        if (!got) {
          ok = false;
          break;
        }
        g.issue(smem_u32(sA + stage * A_BYTES), kb);
        cp_async_arrive_noinc(gfull0 + 8 * stage);
        if (++stage == STAGES) {
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
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < num_kb; ++kb) {
          if (stage % kForwarders == fwd) {
            if (!mbar_wait(gfull0 + 8 * stage, phase, s_abort, a.timeout_ns)) {
              ok = false;
              break;
            }
            fence_proxy_async_smem();
            mbar_arrive(full0 + 8 * stage);
          }
          if (++stage == STAGES) {
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
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            umma_bf16(d_tmem, sw128_desc(a_addr + k * UMMA_K * 2), sw128_desc(b_addr + k * UMMA_K * 2), idesc,
                      (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(empty0 + 8 * stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull0 + 8 * acc);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutMma);
        *s_abort = 1;
      }
      // all MMAs issued by this thread have finished once `drain` completes
      umma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, a.timeout_ns);
    }
  } else if (warp < 6) {
    // -------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileCoord c = decode_tile(tile, s_mstart, E, a.n_tiles);
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      const int row = s_offsets[c.e] + c.m * BM + q * 32 + lane;
      const bool valid = row < s_offsets[c.e] + s_counts[c.e];
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (EPI == kEpiSwiGLU) {
        // columns [0,128) = gate, [128,256) = up, for H columns n*128 .. n*128+127
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(row) * a.ldo + c.n * (BN / 2);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t g[32], u[32];
          tmem_ld32_sync(tbase + ch * 32, g);
          tmem_ld32_sync(tbase + 128 + ch * 32, u);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            const float h0 = silu_fast(g0) * u0;
            const float h1 = silu_fast(g1) * u1;
            p[i] = pack_bf16(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
          }
        }
      } else if constexpr (EPI == kEpiReluBias) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(row) * a.ldo + c.n * BN;
        const float* bias = a.bias + static_cast<size_t>(c.e) * a.out_cols + c.n * BN;
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h0 = fmaxf(__uint_as_float(v[2 * i]) + bias[ch * 32 + 2 * i], 0.f);
            const float h1 = fmaxf(__uint_as_float(v[2 * i + 1]) + bias[ch * 32 + 2 * i + 1], 0.f);
            p[i] = pack_bf16(h0, h1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(out + ch * 32);
#pragma unroll
            for (int w = 0; w < 4; ++w) dst[w] = make_uint4(p[4 * w], p[4 * w + 1], p[4 * w + 2], p[4 * w + 3]);
          }
        }
      } else if constexpr (EPI == kEpiCombineF32) {
        // out[token] += gate * (acc (+ b2)): with two slots and a zeroed output the two reductions give
        // RN(g0*y0 + g1*y1) in either order, the value the separate combine computes
        const int tok = valid ? a.token_of_row[row] : 0;
        const float gr = valid ? a.gate_of_row[row] : 0.f;
        float* out = static_cast<float*>(a.out) + static_cast<size_t>(tok) * a.ldo + c.n * BN;
        const float* bias = a.bias ? a.bias + static_cast<size_t>(c.e) * a.out_cols + c.n * BN : nullptr;
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          if (valid) {
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              float y[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                y[i] = __uint_as_float(v[4 * w + i]);
                if (bias) y[i] += bias[ch * 32 + 4 * w + i];
                y[i] = __fmul_rn(gr, y[i]);
              }
              red_add_v4(out + ch * 32 + 4 * w, y[0], y[1], y[2], y[3]);
            }
          }
        }
      } else {
        float* out = static_cast<float*>(a.out) + static_cast<size_t>(row) * a.ldo + c.n * BN;
        const float* bias = a.bias ? a.bias + static_cast<size_t>(c.e) * a.out_cols + c.n * BN : nullptr;
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          tmem_ld32_sync(tbase + ch * 32, v);
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(out + ch * 32);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              float4 o = make_float4(__uint_as_float(v[4 * w]), __uint_as_float(v[4 * w + 1]),
                                     __uint_as_float(v[4 * w + 2]), __uint_as_float(v[4 * w + 3]));
              if (bias) {
                o.x += bias[ch * 32 + 4 * w];
                o.y += bias[ch * 32 + 4 * w + 1];
                o.z += bias[ch * 32 + 4 * w + 2];
                o.w += bias[ch * 32 + 4 * w + 3];
              }
              dst[w] = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
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
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int EPI, bool GA>
cudaError_t launch_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid, cudaStream_t s) {
  const int threads = GA ? NUM_THREADS_GA : (a.zero_out ? NUM_THREADS_ZERO : NUM_THREADS);
  return pdl_launch(tc_grouped_gemm_kernel<EPI, GA>, dim3(grid), dim3(threads), SMEM_BYTES, s, tmA, tmB, a);
}

template <int EPI, bool GA>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(tc_grouped_gemm_kernel<EPI, GA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_BYTES);
}

}  // namespace

cudaError_t prepare_tc_gemm() {
  cudaError_t e = set_smem<kEpiSwiGLU, false>();
  if (e == cudaSuccess) e = set_smem<kEpiSwiGLU, true>();
  if (e == cudaSuccess) e = set_smem<kEpiReluBias, false>();
  if (e == cudaSuccess) e = set_smem<kEpiReluBias, true>();
  if (e == cudaSuccess) e = set_smem<kEpiStoreF32, false>();
  if (e == cudaSuccess) e = set_smem<kEpiCombineF32, false>();
  return e;
}

int tc_gemm_block_n() { return BN; }
int tc_gemm_threads() { return NUM_THREADS; }

// gather_a: A rows are gathered from a.gather_x through a.token_of_row (up-projection epilogues
// only) and tmA is not read.
cudaError_t launch_tc_gemm(int epi, bool gather_a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const GemmArgs& a, int grid, cudaStream_t s) {
  if (grid <= 0) return cudaSuccess;
  switch (epi) {
    case kEpiSwiGLU:
      return gather_a ? launch_t<kEpiSwiGLU, true>(tmA, tmB, a, grid, s) : launch_t<kEpiSwiGLU, false>(tmA, tmB, a, grid, s);
    case kEpiReluBias:
      return gather_a ? launch_t<kEpiReluBias, true>(tmA, tmB, a, grid, s)
                      : launch_t<kEpiReluBias, false>(tmA, tmB, a, grid, s);
    case kEpiCombineF32:
      if (gather_a) return cudaErrorInvalidValue;
      return launch_t<kEpiCombineF32, false>(tmA, tmB, a, grid, s);
    default:
      if (gather_a) return cudaErrorInvalidValue;
      return launch_t<kEpiStoreF32, false>(tmA, tmB, a, grid, s);
  }
}

}  // namespace colibri
