// Decode-sized batches (T <= 64): expert FFN as weight-streaming tcgen05 GEMMs.
//
// With a few tokens per expert the layer is bound by reading the weights of the experts that
// received tokens (zskr.cn/news/2272131 "Colibri: a lightweight C MoE inference engine for edge
// devices" 2.2: only the routed experts' weights are touched; 2.1 Compute: grouped GEMM per expert).
// So the roles of the operands are swapped: the weight rows are the M = 128 side of the MMA and the
// expert's token rows (padded to n_pad = 16..64) are the N side:
//
//   P[s][tok][row] = sum over k in split s of  W_e[row, k] * X_e[tok, k]     (fp32, TMEM)
//
// Work items are (active expert, 128-row weight tile, K split), spread over one persistent CTA per
// SM, so every weight byte is read once and all SMs stream.  The number of K splits S is chosen on
// the device from the expert counts (the same pure function in every kernel) so items fill whole
// waves.  Partial sums are reduced in split order -- deterministic -- by
//   decode_act_kernel      up projection: sum splits, SwiGLU (or +b1, ReLU) -> H rows (bf16)
//   decode_combine_kernel  down projection: sum splits (+b2), gate-weighted combine -> out
// Warp roles, barriers and bounded waits are those of the prefill grouped GEMM.
#include "tcgen05_ptx.cuh"

namespace colibri {
namespace {

using namespace ptx;

constexpr int DBM = 128, DBK = 64, DUMMA_K = 16;
constexpr int DSTAGES = 8;
constexpr int DA_BYTES = DBM * DBK * 2;      // 16 KB weight tile
constexpr int DB_SLOT = kDecodeSepMaxT * DBK * 2;  // 8 KB token-tile slot (n_pad rows used)
constexpr int DNUM_THREADS = 192;
constexpr uint32_t DTMEM_COLS = 128;           // two accumulators of up to 64 fp32 columns
constexpr int DNUM_BARS = 2 * DSTAGES + 5;
constexpr int DSMEM_BYTES = 1024 + DSTAGES * (DA_BYTES + DB_SLOT) + DNUM_BARS * 8 + 16 + 4 * (3 * kMaxE + 2);
static_assert(DSMEM_BYTES <= 227 * 1024, "decode GEMM shared memory");

__global__ void __launch_bounds__(DNUM_THREADS, 1)
    tc_decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                          const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + DSTAGES * DA_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + DSTAGES * DB_SLOT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + DNUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_counts = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_offsets = s_counts + kMaxE;
  int* s_act = s_offsets + kMaxE + 1;
  int* s_nact = s_act + kMaxE;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + DSTAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * DSTAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * DSTAGES + 2);
  const uint32_t drain = smem_u32(bars + 2 * DSTAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  pdl_trigger();
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < DSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull0 + 8 * i, 1);
      mbar_init(tempty0 + 8 * i, 4);
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), DTMEM_COLS);
    tmem_relinquish();
  }
  // The routing summary (Sched) comes from the router, two or more kernels back.  The kernel right
  // before this one triggers its dependents only after its own griddepcontrol.wait, so this grid
  // starts after the router has finished and may read Sched before waiting.  The token rows (Xp or
  // H) and the partial-sum buffer belong to the kernel right before: touched only after pdl_wait.
  if (threadIdx.x < kMaxE) s_counts[threadIdx.x] = threadIdx.x < E ? a.sched->counts[threadIdx.x] : 0;
  if (threadIdx.x < kMaxE + 1) s_offsets[threadIdx.x] = threadIdx.x <= E ? a.sched->offsets[threadIdx.x] : 0;
  if (threadIdx.x == 0) *s_nact = active_experts(a.sched, E, s_act);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int n_act = *s_nact;
  const int MT = a.n_per_expert / DBM;
  const int KB = (a.K + DBK - 1) / DBK;
  const int S = decode_splits(n_act * MT, KB, a.grid_ref, a.s_max);
  const int total = n_act * MT * S;
  const int n_pad = a.n_pad;
  const uint32_t b_bytes = static_cast<uint32_t>(n_pad) * DBK * 2;

  if (!(warp == 0 && lane == 0)) pdl_wait();
  if (warp == 0) {
    if (lane == 0) {
      // The weights do not depend on the previous kernel: the weight tiles of the first DSTAGES
      // stages are requested before waiting for it (their full barriers expect the token bytes too)
      int pre = 0;
      for (int it = blockIdx.x; pre < DSTAGES && it < total; it += gridDim.x) {
        const int ai = it / (MT * S), r = it - ai * (MT * S), mt = r / S, sp = r - (r / S) * S;
        const int kb0 = (KB * sp) / S, kb1 = (KB * (sp + 1)) / S;
        const int w_row = s_act[ai] * a.n_per_expert + mt * DBM;
        for (int kb = kb0; kb < kb1 && pre < DSTAGES; ++kb, ++pre) {
          mbar_arrive_expect_tx(full0 + 8 * pre, DA_BYTES + b_bytes);
          tma_load_2d(smem_u32(sA + pre * DA_BYTES), &tmW, full0 + 8 * pre, kb * DBK, w_row);
        }
      }
      pdl_wait();
      int stage = 0, g = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
        const int ai = it / (MT * S), r = it - ai * (MT * S), mt = r / S, sp = r - (r / S) * S;
        const int e = s_act[ai];
        const int kb0 = (KB * sp) / S, kb1 = (KB * (sp + 1)) / S;
        const int w_row = e * a.n_per_expert + mt * DBM;
        const int x_row = s_offsets[e];
        for (int kb = kb0; kb < kb1; ++kb, ++g) {
          if (g >= pre) {  // stages before `pre` are in their first round: free, weights in flight
            if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, s_abort, a.timeout_ns)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(full0 + 8 * stage, DA_BYTES + b_bytes);
            tma_load_2d(smem_u32(sA + stage * DA_BYTES), &tmW, full0 + 8 * stage, kb * DBK, w_row);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          tma_load_2d(smem_u32(sB + stage * DB_SLOT), &tmX, full0 + 8 * stage, kb * DBK, x_row);
          if (++stage == DSTAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
        *s_abort = 1;
      }
      for (int s = 0; s < DSTAGES; ++s)
        if (armed & (1u << s)) {
          volatile int never = 0;
          mbar_wait(full0 + 8 * s, (armed_phase >> s) & 1u, &never, a.timeout_ns);
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16(DBM, n_pad);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
        const int r = it % (MT * S), sp = r % S;
        const int kb0 = (KB * sp) / S, kb1 = (KB * (sp + 1)) / S;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kDecodeSepMaxT);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * DA_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * DB_SLOT);
#pragma unroll
          for (int k = 0; k < DBK / DUMMA_K; ++k)
            umma_bf16(d_tmem, sw128_desc(a_addr + k * DUMMA_K * 2), sw128_desc(b_addr + k * DUMMA_K * 2), idesc,
                      (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(empty0 + 8 * stage);
          if (++stage == DSTAGES) {
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
      umma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, a.timeout_ns);
    }
  } else {
    // epilogue: thread = weight row of the tile, 16 token columns per TMEM load
    const int q = warp & 3;
    const size_t rows_total = static_cast<size_t>(E) * a.n_per_expert;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
      const int ai = it / (MT * S), r = it - ai * (MT * S), mt = r / S, sp = r - (r / S) * S;
      const int e = s_act[ai];
      const int cnt = s_counts[e];
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      const size_t row = static_cast<size_t>(e) * a.n_per_expert + mt * DBM + q * 32 + lane;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kDecodeSepMaxT);
      float* P = a.partial + static_cast<size_t>(sp) * n_pad * rows_total + row;
      for (int c = 0; c < n_pad; c += 16) {
        uint32_t v[16];
        tmem_ld16_sync(tbase + c, v);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c + j < cnt) P[static_cast<size_t>(c + j) * rows_total] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, DTMEM_COLS);
  }
}

// Up projection: H[offsets[e] + tok, c] = act(sum_s P[s][tok][rows of c]), one thread per 4 columns.
template <bool kSwiGLU>
__global__ void __launch_bounds__(256) decode_act_kernel(DecodeActArgs a) {
  __shared__ int s_act[kMaxE];
  __shared__ int s_S;
  const int e = blockIdx.y;
  pdl_wait();
  pdl_trigger();  // after the wait: the down GEMM reads the router's summary before its own wait
  const int cnt = a.sched->counts[e];
  if (cnt == 0) return;
  if (threadIdx.x == 0) {
    const int n_act = active_experts(a.sched, a.E, s_act);
    s_S = decode_splits(n_act * (a.n_per_expert / DBM), (a.K + DBK - 1) / DBK, a.grid_ref, a.s_max);
  }
  __syncthreads();
  const int S = s_S;
  const int f = a.f, f4 = f / 4;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int tok = idx / f4, c = (idx - tok * f4) * 4;
  if (tok >= cnt) return;
  const size_t rows_total = static_cast<size_t>(a.E) * a.n_per_expert;
  float h[4];
  if constexpr (kSwiGLU) {
    const size_t grow = static_cast<size_t>(e) * a.n_per_expert + 256 * (c / 128) + (c % 128);
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int s = 0; s < S; ++s) {
      const float* P = a.partial + (static_cast<size_t>(s) * a.n_pad + tok) * rows_total;
      const float4 pg = *reinterpret_cast<const float4*>(P + grow);
      const float4 pu = *reinterpret_cast<const float4*>(P + grow + 128);
      g.x += pg.x; g.y += pg.y; g.z += pg.z; g.w += pg.w;
      u.x += pu.x; u.y += pu.y; u.z += pu.z; u.w += pu.w;
    }
    h[0] = silu_fast(g.x) * u.x;
    h[1] = silu_fast(g.y) * u.y;
    h[2] = silu_fast(g.z) * u.z;
    h[3] = silu_fast(g.w) * u.w;
  } else {
    const size_t grow = static_cast<size_t>(e) * a.n_per_expert + c;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float4 p = *reinterpret_cast<const float4*>(a.partial + (static_cast<size_t>(s) * a.n_pad + tok) *
                                                                        rows_total + grow);
      v.x += p.x; v.y += p.y; v.z += p.z; v.w += p.w;
    }
    const float* b = a.bias + static_cast<size_t>(e) * f + c;
    h[0] = fmaxf(v.x + b[0], 0.f);
    h[1] = fmaxf(v.y + b[1], 0.f);
    h[2] = fmaxf(v.z + b[2], 0.f);
    h[3] = fmaxf(v.w + b[3], 0.f);
  }
  uint2 o;
  o.x = pack_bf16(h[0], h[1]);
  o.y = pack_bf16(h[2], h[3]);
  *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.h) +
                            static_cast<size_t>(a.sched->offsets[e] + tok) * f + c) = o;
}

// Down projection + combine: out[t, c] = sum over the token's slots k, in order, of
// g_k * (sum over K splits of P[split][row slot][e_k rows] (+ b2)).
template <bool kBf16Out>
__global__ void __launch_bounds__(256) decode_combine_kernel(DecodeCombineArgs a) {
  __shared__ int s_act[kMaxE];
  __shared__ int s_S;
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    const int n_act = active_experts(a.sched, a.E, s_act);
    s_S = decode_splits(n_act * (a.d / DBM), (a.K + DBK - 1) / DBK, a.grid_ref, a.s_max);
  }
  __syncthreads();
  const int S = s_S;
  const int t = blockIdx.y;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (c >= a.d) return;
  const size_t rows_total = static_cast<size_t>(a.E) * a.d;
  const int Sl = a.S;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kMaxSlots; ++k) {
    if (k >= Sl) break;
    const int e = a.idx[Sl * t + k];
    const int slot = a.row_of[Sl * t + k] - a.sched->offsets[e];
    const size_t grow = static_cast<size_t>(e) * a.d + c;
    // all splits' partials requested before the (split-ordered) sum
    float4 p[kDecodeSplitsDown];
#pragma unroll
    for (int s = 0; s < kDecodeSplitsDown; ++s)
      p[s] = s < S ? *reinterpret_cast<const float4*>(a.partial + (static_cast<size_t>(s) * a.n_pad + slot) *
                                                                      rows_total + grow)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v = p[0];
#pragma unroll
    for (int s = 1; s < kDecodeSplitsDown; ++s)
      if (s < S) {
        v.x += p[s].x; v.y += p[s].y; v.z += p[s].z; v.w += p[s].w;
      }
    if (a.bias) {
      const float* b = a.bias + grow;
      v.x += b[0]; v.y += b[1]; v.z += b[2]; v.w += b[3];
    }
    const float gk = a.gate[Sl * t + k];
    const float y[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = k == 0 ? __fmul_rn(gk, y[i]) : __fadd_rn(o[i], __fmul_rn(gk, y[i]));
  }
  if constexpr (kBf16Out) {
    uint2 p;
    p.x = pack_bf16(o[0], o[1]);
    p.y = pack_bf16(o[2], o[3]);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(t) * a.d + c) = p;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<size_t>(t) * a.d + c) =
        make_float4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t prepare_decode_gemm() {
  return cudaFuncSetAttribute(tc_decode_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DSMEM_BYTES);
}

cudaError_t launch_decode_gemm(const CUtensorMap& tmW, const CUtensorMap& tmX, const DecodeArgs& a, int grid,
                               cudaStream_t s) {
  return pdl_launch(tc_decode_gemm_kernel, dim3(grid), dim3(DNUM_THREADS), DSMEM_BYTES, s, tmW, tmX, a);
}

cudaError_t launch_decode_act(bool swiglu, const DecodeActArgs& a, cudaStream_t s) {
  const int per_expert = a.n_pad * (a.f / 4);
  dim3 grid((per_expert + 255) / 256, a.E);
  if (swiglu) return pdl_launch(decode_act_kernel<true>, grid, dim3(256), 0, s, a);
  return pdl_launch(decode_act_kernel<false>, grid, dim3(256), 0, s, a);
}

cudaError_t launch_decode_combine(int out_dtype, const DecodeCombineArgs& a, cudaStream_t s) {
  dim3 grid((a.d / 4 + 255) / 256, a.T);
  if (out_dtype == 0) return pdl_launch(decode_combine_kernel<false>, grid, dim3(256), 0, s, a);
  return pdl_launch(decode_combine_kernel<true>, grid, dim3(256), 0, s, a);
}

}  // namespace colibri
