// Decode-sized batches (T <= 128) in one cooperative kernel: up projection, activation, down
// projection and combine, separated by grid-wide barriers instead of kernel boundaries.
//
// What is computed is the separate-kernel decode path's (gemm_decode.cu: the Compute stage of
// zskr.cn/news/2272131 "Colibri: a lightweight C MoE inference engine for edge devices" 2.1 as a
// stream over the weights of the experts that received tokens, 2.2), reorganised for latency:
//
//   phase U  P[s][t][e rows] = sum over K split s of W13_e[rows, k] x[t, k]   (tcgen05, TMEM)
//   phase A  H[e * n_pad + t, :] = act(sum_s P[s][t][e rows])  for every routed (token, expert)
//            -- or, when phase U runs unsplit (S = 1, the usual case), phase U's epilogue writes H
//            itself and phase A and its barrier drop out: its weight tiles are then two 64-row
//            boxes, the gate rows of 64 hidden units and their up rows, so the warps holding the
//            up values hand them to the warps holding the gates through shared memory
//   phase D  P[s][t][e rows] = sum over split s of W2_e[rows, k] H[e * n_pad + t, k]
//   phase C  out[t, :] = sum over t's slots in order of g * (sum_s P[s][t][e rows] (+ b2)): after a
//            third barrier, or (tile_combine, the smallest batches) for the 128 columns of a down-
//            projection weight tile by the CTA that finished the tile's last item (a per-tile
//            counter, reset by that CTA), with no barrier.  The counter costs a gpu-scope fence per
//            item, which only pays off while items are few and each combine is a handful of rows.
//
// The token operand of phase U is x itself (all n_pad >= T token rows of the batch, rows past T
// read as zeros by TMA), so no dispatch copy is needed: a column t of expert e's accumulator is
// kept only when t was routed to e (a 128-bit token mask per expert).  One persistent CTA per SM,
// the warp roles of the decode GEMM (TMA producer, MMA issuer, 4 epilogue warps); every thread
// joins the element-wise phase A.  The weight tiles of phase D are requested before the barriers
// that precede it (they do not depend on phase A), so the HBM stream continues across them.
//
// Barriers: one arrival per CTA on a counter in the routing summary (cleared by the router), a
// gpu-scope release, then a spin on acquire loads bounded by the wait timeout; H is written through the generic proxy and read by TMA, so its writers fence the proxy
// before arriving.  Splits are summed in order: results are deterministic.
#include "tcgen05_ptx.cuh"

namespace colibri {
namespace {

using namespace ptx;

constexpr int FBM = 128, FBK = 64, FUMMA_K = 16;
// The ring: FSTAGES_MAX stages of a 16 KB weight tile and an 8 KB token slot (n_pad <= 64), or six
// stages with a 16 KB token slot for 65..128 tokens.
constexpr int FSTAGES_MAX = 8;
constexpr int FRING_BYTES = 192 * 1024;
constexpr int FA_BYTES = FBM * FBK * 2;          // 16 KB weight tile
constexpr int FNUM_THREADS = 192;
constexpr uint32_t FTMEM_COLS = 2 * kDecodeMaxT;  // two accumulators of up to 128 fp32 columns
constexpr int FNUM_BARS = 2 * FSTAGES_MAX + 5;
constexpr int FHALF = FBM / 2;                   // hidden units per weight tile with SwiGLU (direct H)
constexpr int FX_CHUNK = 16;                     // token columns per TMEM load
constexpr int FX_BYTES = 2 * FX_CHUNK * FHALF * 4;  // up values handed over: two buffers of 16 x 64
constexpr int FSMEM_BYTES =
    1024 + FRING_BYTES + FX_BYTES + FNUM_BARS * 8 + 16 + 16 * kMaxE + 4 * (2 * kMaxE + 4);
static_assert(FSMEM_BYTES <= 227 * 1024, "fused decode shared memory");

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The four epilogue warps (2..5) only.
__device__ __forceinline__ void named_barrier_epilogue() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Same barrier, and the AND of `v` over the four epilogue warps (so they all stop or go on together).
__device__ __forceinline__ bool epilogue_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// Grid-wide barrier number `n` (1, 2, ...): every CTA arrives once; bounded wait.  The arrival is a
// gpu-scope release (it covers the CTA's writes, ordered before it by the CTA barrier) and the spin an
// acquire; the closing CTA barrier orders every thread's later reads after that acquire.
__device__ __forceinline__ void grid_barrier(Sched* sc, uint32_t n, volatile int* s_abort, uint64_t timeout_ns,
                                             int32_t* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&sc->grid_sync) : "memory");
    const uint32_t target = n * gridDim.x;
    if (ld_acquire_gpu(&sc->grid_sync) < target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(&sc->grid_sync) < target) {
        if (globaltimer_ns() - t0 > timeout_ns) {
          atomicOr(status, kStatusTimeoutGridSync);
          *s_abort = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
}

// One weight-streaming GEMM phase: items (active expert, 128-row weight tile, K split).
struct Phase {
  const CUtensorMap* tmW;
  const CUtensorMap* tmX;
  int K;        // reduction length
  int rows;     // weight rows per expert
  int x_step;   // first token row of expert e's operand = e * x_step
  int MT, KB, S, total;
  float* partial;  // [S][n_pad][E * rows]
  const CUtensorMap* tmWh;  // direct H: the same weights in 64-row boxes, else nullptr
  bool direct;              // phase U writes H (S == 1)
};

__device__ __forceinline__ Phase make_phase(const CUtensorMap* tmW, const CUtensorMap* tmX, int K, int rows, int x_step,
                                            int n_act, int s_max, float* partial) {
  Phase p;
  p.tmW = tmW;
  p.tmX = tmX;
  p.K = K;
  p.rows = rows;
  p.x_step = x_step;
  p.MT = rows / FBM;
  p.KB = (K + FBK - 1) / FBK;
  p.S = decode_splits(n_act * p.MT, p.KB, gridDim.x, s_max);
  p.total = n_act * p.MT * p.S;
  p.partial = partial;
  p.tmWh = nullptr;
  p.direct = false;
  return p;
}

struct Item {
  int e, mt, sp, kb0, kb1;
};
__device__ __forceinline__ Item item_of(const Phase& p, int it, const int* s_act) {
  Item r;
  const int ai = it / (p.MT * p.S), rem = it - ai * (p.MT * p.S);
  r.e = s_act[ai];
  r.mt = rem / p.S;
  r.sp = rem - r.mt * p.S;
  r.kb0 = (p.KB * r.sp) / p.S;
  r.kb1 = (p.KB * (r.sp + 1)) / p.S;
  return r;
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  int n = FSTAGES_MAX;  // stages in the ring
  __device__ __forceinline__ void next() {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

__global__ void __launch_bounds__(FNUM_THREADS, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tmW13, const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ CUtensorMap tmW13h, const FusedDecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xs = reinterpret_cast<float*>(smem + FRING_BYTES);  // [2][16 tokens][64 units] (direct H)
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xs) + FX_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + FNUM_BARS);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // tokens routed to e: bit t of the 128-bit mask s_mask[2e] | s_mask[2e + 1] << 64
  unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(tmem_slot + 4);
  int* s_act = reinterpret_cast<int*>(s_mask + 2 * kMaxE);
  int* s_nact = s_act + kMaxE;
  volatile int* s_last = s_nact + 1;  // this CTA completed the current weight tile (phase D)

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + FSTAGES_MAX);
  const uint32_t tfull0 = smem_u32(bars + 2 * FSTAGES_MAX);
  const uint32_t tempty0 = smem_u32(bars + 2 * FSTAGES_MAX + 2);
  const uint32_t drain = smem_u32(bars + 2 * FSTAGES_MAX + 4);
  // ring geometry: stage s holds the weight tile at +0 and the token tile at +16 KB
  const int stride = a.n_pad <= 64 ? FA_BYTES + 8 * 1024 : FA_BYTES + 16 * 1024;
  const int nst = FRING_BYTES / stride;  // 8 or 6
  auto stage_a = [&](int st) { return smem_u32(smem + st * stride); };
  auto stage_b = [&](int st) { return smem_u32(smem + st * stride + FA_BYTES); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, T = a.T, Sl = a.S, n_pad = a.n_pad;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < FSTAGES_MAX; ++s) {
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
    prefetch_tmap(&tmW13);
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW2);
    prefetch_tmap(&tmH);
    prefetch_tmap(&tmW13h);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), FTMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x < 2 * kMaxE) s_mask[threadIdx.x] = 0ull;
  pdl_trigger();
  pdl_wait();  // routing (idx, gates, counts) comes from the router
  // every routing load of this thread in flight at once (T * S <= 640 slots, E <= 17 counts)
  constexpr int kSlotLoads = 4;
  static_assert(kSlotLoads * FNUM_THREADS >= kDecodeMaxT * kMaxSlots, "routing slots per thread");
  const int n_slots = T * Sl;
  int ev[kSlotLoads];
#pragma unroll
  for (int u = 0; u < kSlotLoads; ++u) {
    const int i = threadIdx.x + u * FNUM_THREADS;
    ev[u] = i < n_slots ? a.idx[i] : -1;
  }
  const int cnt = threadIdx.x < E ? a.sched->counts[threadIdx.x] : 0;
  __syncthreads();  // masks cleared
#pragma unroll
  for (int u = 0; u < kSlotLoads; ++u) {
    const int i = threadIdx.x + u * FNUM_THREADS, t = i / Sl;
    if (ev[u] >= 0 && ev[u] < E) atomicOr(&s_mask[2 * ev[u] + (t >> 6)], 1ull << (t & 63));
  }
  if (warp == 0) {  // active experts in index order, from the counts
    const unsigned act = __ballot_sync(0xffffffffu, lane < E && cnt > 0);
    if (lane < E && cnt > 0) s_act[__popc(act & ((1u << lane) - 1u))] = lane;
    if (lane == 0) *s_nact = __popc(act);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_act = *s_nact;
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x, gstride = gridDim.x * blockDim.x;
  const uint32_t b_bytes = static_cast<uint32_t>(n_pad) * FBK * 2;
  const uint32_t idesc = make_idesc_bf16(FBM, n_pad);

  Phase PU = make_phase(&tmW13, &tmX, a.d, a.n_up, 0, n_act, kDecodeSplitsUp, a.partial);
  if (a.direct_h && PU.S == 1) {
    PU.tmWh = &tmW13h;
    PU.direct = true;
  }
  const Phase PD = make_phase(&tmW2, &tmH, a.f, a.d, n_pad, n_act, kDecodeSplitsDown, a.partial);

  // per-role state, carried from phase U to phase D
  Ring ring;                         // producer and MMA issuer: shared-memory ring position
  ring.n = nst;
  int acc = 0;                       // MMA issuer and epilogue: TMEM accumulator in use
  uint32_t acc_phase = 0;
  uint32_t armed = 0, armed_phase = 0;  // producer: stages with copies issued (last phase of each)
  int pre = 0;                       // producer: stages of phase D whose weight tile is in flight
  Ring pre_start;

  // The weight tile of item im at K block kb: one 128-row box, or (direct H with SwiGLU) the gate
  // rows 256*(mt/2) + 64*(mt%2) + [0, 64) and the up rows 128 further on, in two 64-row boxes.
  auto load_weights = [&](const Phase& P, const Item& im, uint32_t dst, uint32_t bar, int kb) {
    if (P.direct) {
      const int r0 = im.e * P.rows + (a.swiglu ? 2 * FBM * (im.mt >> 1) + FHALF * (im.mt & 1) : FBM * im.mt);
      const int r1 = r0 + (a.swiglu ? FBM : FHALF);
      tma_load_2d(dst, P.tmWh, bar, kb * FBK, r0);
      tma_load_2d(dst + FHALF * FBK * 2, P.tmWh, bar, kb * FBK, r1);
    } else {
      tma_load_2d(dst, P.tmW, bar, kb * FBK, im.e * P.rows + im.mt * FBM);
    }
  };
  // Producer: weight tile + token tile per stage.  Stages [0, pre) of this phase had their weight
  // tile requested earlier (from pre_start on); only their token tile is issued here.
  auto produce = [&](const Phase& P, int n_pre, Ring start) {
    Ring cur = n_pre > 0 ? start : ring;
    int g = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < P.total; it += gridDim.x) {
      const Item im = item_of(P, it, s_act);
      const int x_row = im.e * P.x_step;
      for (int kb = im.kb0; kb < im.kb1; ++kb, ++g) {
        const uint32_t fb = full0 + 8 * cur.stage;
        if (g >= n_pre) {
          if (!mbar_wait(empty0 + 8 * cur.stage, cur.phase ^ 1u, s_abort, a.timeout_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(fb, FA_BYTES + b_bytes);
          load_weights(P, im, stage_a(cur.stage), fb, kb);
        }
        armed |= 1u << cur.stage;
        armed_phase = (armed_phase & ~(1u << cur.stage)) | (cur.phase << cur.stage);
        tma_load_2d(stage_b(cur.stage), P.tmX, fb, kb * FBK, x_row);
        cur.next();
      }
    }
    if (!ok) {
      if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
      *s_abort = 1;
    }
    ring = cur;
  };
  // Producer: request the weight tiles of phase P's first stages (its token operand is not ready).
  auto prefetch_weights = [&](const Phase& P) {
    pre_start = ring;
    pre = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && pre < nst && it < P.total; it += gridDim.x) {
      const Item im = item_of(P, it, s_act);
      for (int kb = im.kb0; kb < im.kb1 && pre < nst; ++kb, ++pre) {
        if (!mbar_wait(empty0 + 8 * ring.stage, ring.phase ^ 1u, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * ring.stage;
        mbar_arrive_expect_tx(fb, FA_BYTES + b_bytes);
        load_weights(P, im, stage_a(ring.stage), fb, kb);
        ring.next();
      }
    }
    if (!ok) {
      if (!*s_abort) atomicOr(a.status, kStatusTimeoutProducer);
      *s_abort = 1;
    }
  };
  auto mma = [&](const Phase& P) {
    bool ok = true;
    for (int it = blockIdx.x; ok && it < P.total; it += gridDim.x) {
      const Item im = item_of(P, it, s_act);
      if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, s_abort, a.timeout_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kDecodeMaxT);
      for (int kb = im.kb0; kb < im.kb1; ++kb) {
        if (!mbar_wait(full0 + 8 * ring.stage, ring.phase, s_abort, a.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = stage_a(ring.stage);
        const uint32_t b_addr = stage_b(ring.stage);
#pragma unroll
        for (int k = 0; k < FBK / FUMMA_K; ++k)
          umma_bf16(d_tmem, sw128_desc(a_addr + k * FUMMA_K * 2), sw128_desc(b_addr + k * FUMMA_K * 2), idesc,
                    (kb > im.kb0 || k > 0) ? 1u : 0u);
        umma_commit(empty0 + 8 * ring.stage);
        ring.next();
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
  };
  // Phase D's combine, for the 128 output columns of weight tile mt, by the CTA whose item completed
  // that tile last (all experts' splits of those rows are then in the partial buffer).
  auto combine_tile = [&](const Phase& P, int mt) {
    const int d = a.d;
    const size_t rows_total = static_cast<size_t>(E) * d;
    const int et = threadIdx.x - 64;  // epilogue thread 0..127
    for (int w = et; w < T * (FBM / 4); w += 128) {
      const int t = w / (FBM / 4), c = mt * FBM + (w - t * (FBM / 4)) * 4;
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k = 0; k < Sl; ++k) {
        const int e = a.idx[t * Sl + k];
        const size_t grow = static_cast<size_t>(e) * d + c;
        float4 p[kDecodeSplitsDown];
#pragma unroll
        for (int sp = 0; sp < kDecodeSplitsDown; ++sp)
          p[sp] = sp < P.S ? __ldcg(reinterpret_cast<const float4*>(a.partial + (static_cast<size_t>(sp) * n_pad + t) *
                                                                                rows_total + grow))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 v = p[0];
#pragma unroll
        for (int sp = 1; sp < kDecodeSplitsDown; ++sp)
          if (sp < P.S) {
            v.x += p[sp].x; v.y += p[sp].y; v.z += p[sp].z; v.w += p[sp].w;
          }
        if (a.b2) {
          const float* b = a.b2 + grow;
          v.x += b[0]; v.y += b[1]; v.z += b[2]; v.w += b[3];
        }
        const float gk = a.gate[t * Sl + k];
        const float y[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = k == 0 ? __fmul_rn(gk, y[i]) : __fadd_rn(o[i], __fmul_rn(gk, y[i]));
      }
      if (a.out_bf16) {
        uint2 pk;
        pk.x = pack_bf16(o[0], o[1]);
        pk.y = pack_bf16(o[2], o[3]);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(t) * d + c) = pk;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<size_t>(t) * d + c) =
            make_float4(o[0], o[1], o[2], o[3]);
      }
    }
  };

  // Epilogue: thread = weight row of the item's tile; token column t kept when t was routed to e.
  // With `combine`, each item then counts itself done for its weight tile; the CTA completing the
  // tile's last item (every active expert, every split) combines that tile's output columns.
  auto epilogue = [&](const Phase& P, bool combine) {
    const int q = warp & 3;
    const int wr = q * 32 + lane;  // weight row of the tile
    const size_t rows_total = static_cast<size_t>(E) * P.rows;
    int xb = 0;
    for (int it = blockIdx.x; it < P.total; it += gridDim.x) {
      const Item im = item_of(P, it, s_act);
      const unsigned long long mlo = s_mask[2 * im.e], mhi = s_mask[2 * im.e + 1];
      // token columns c .. c + 15 of the mask (16-column chunks never straddle its two words)
      auto mask16 = [&](int c) -> unsigned long long { return c < 64 ? mlo >> c : mhi >> (c - 64); };
      bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, s_abort, a.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (combine || (P.direct && a.swiglu)) ok = epilogue_all(ok);  // named barriers below need all four warps
      if (!ok) {
        if (lane == 0 && !*s_abort) atomicOr(a.status, kStatusTimeoutEpilogue);
        if (lane == 0) *s_abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kDecodeMaxT);
      if (P.direct) {
        // H rows e * n_pad + t of the routed tokens, written here (phase A is skipped)
        __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(a.h) + static_cast<size_t>(im.e) * n_pad * a.f;
        for (int c = 0; c < n_pad; c += FX_CHUNK) {
          uint32_t v[FX_CHUNK];
          tmem_ld16_sync(tbase + c, v);
          if (a.swiglu) {
            // rows 0-63: gates of hidden units 64*mt + [0, 64); rows 64-127: their up values
            float* x = xs + xb * (FX_CHUNK * FHALF);
            if (q >= 2) {
#pragma unroll
              for (int j = 0; j < FX_CHUNK; ++j) x[j * FHALF + wr - FHALF] = __uint_as_float(v[j]);
            }
            named_barrier_epilogue();
            if (q < 2) {
              const int col = im.mt * FHALF + wr;
#pragma unroll
              for (int j = 0; j < FX_CHUNK; ++j)
                if ((mask16(c) >> j) & 1ull)
                  hrow[static_cast<size_t>(c + j) * a.f + col] =
                      __float2bfloat16_rn(silu_fast(__uint_as_float(v[j])) * x[j * FHALF + wr]);
            }
            xb ^= 1;
          } else {
            const int col = im.mt * FBM + wr;
            const float b = a.b1[static_cast<size_t>(im.e) * a.f + col];
#pragma unroll
            for (int j = 0; j < FX_CHUNK; ++j)
              if ((mask16(c) >> j) & 1ull)
                hrow[static_cast<size_t>(c + j) * a.f + col] = __float2bfloat16_rn(fmaxf(__uint_as_float(v[j]) + b, 0.f));
          }
        }
      } else {
        const size_t row = static_cast<size_t>(im.e) * P.rows + im.mt * FBM + wr;
        float* out = P.partial + static_cast<size_t>(im.sp) * n_pad * rows_total + row;
        for (int c = 0; c < n_pad; c += 16) {
          uint32_t v[16];
          tmem_ld16_sync(tbase + c, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if ((mask16(c) >> j) & 1ull) out[static_cast<size_t>(c + j) * rows_total] = __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (combine) {
        named_barrier_epilogue();  // all 128 rows of the item stored
        if (threadIdx.x == 64) {
          __threadfence();
          const uint32_t before = atomicAdd(&a.tile_done[im.mt], 1u);
          const bool last = before == static_cast<uint32_t>(n_act * P.S) - 1u;
          if (last) {
            __threadfence();
            a.tile_done[im.mt] = 0;  // ready for the next forward
          }
          *s_last = last ? 1 : 0;
        }
        named_barrier_epilogue();
        if (*s_last) combine_tile(P, im.mt);
      }
    }
  };

  // ---------------------------------------------------------------- phase U
  if (warp == 0) {
    if (lane == 0) {
      produce(PU, 0, ring);
      prefetch_weights(PD);  // phase D's first weight tiles, independent of phases U and A
    }
  } else if (warp == 1) {
    if (lane == 0) mma(PU);
  } else {
    epilogue(PU, false);
    if (PU.direct) fence_proxy_async_global();  // H is read next by TMA (async proxy)
  }
  uint32_t nbar = 0;  // grid barriers passed
  grid_barrier(a.sched, ++nbar, s_abort, a.timeout_ns, a.status);

  // ---------------------------------------------------------------- phase A: H rows of routed pairs
  if (!PU.direct && !*s_abort) {
    const int f = a.f, f4 = f / 4;
    const size_t rows_total = static_cast<size_t>(E) * a.n_up;
    // kAU work units per thread and round: their partial-sum loads all in flight before any is used
    constexpr int kAU = 4;
    const int n_units = T * Sl * f4;
    for (int w0 = gtid; w0 < n_units; w0 += kAU * gstride) {
      int ue[kAU], ut[kAU], uc[kAU];
      float4 g[kAU], u[kAU];
#pragma unroll
      for (int j = 0; j < kAU; ++j) {
        const int w = w0 + j * gstride;
        const int pair = w < n_units ? w / f4 : 0;
        uc[j] = (w - pair * f4) * 4;
        ut[j] = pair / Sl;
        ue[j] = w < n_units ? a.idx[pair] : -1;
        g[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        u[j] = g[j];
      }
      for (int s = 0; s < PU.S; ++s) {
#pragma unroll
        for (int j = 0; j < kAU; ++j) {
          if (ue[j] < 0) continue;
          const float* P = a.partial + (static_cast<size_t>(s) * n_pad + ut[j]) * rows_total;
          if (a.swiglu) {
            const size_t grow = static_cast<size_t>(ue[j]) * a.n_up + 256 * (uc[j] / 128) + (uc[j] % 128);
            const float4 pg = __ldcg(reinterpret_cast<const float4*>(P + grow));
            const float4 pu = __ldcg(reinterpret_cast<const float4*>(P + grow + 128));
            g[j].x += pg.x; g[j].y += pg.y; g[j].z += pg.z; g[j].w += pg.w;
            u[j].x += pu.x; u[j].y += pu.y; u[j].z += pu.z; u[j].w += pu.w;
          } else {
            const float4 p = __ldcg(reinterpret_cast<const float4*>(P + static_cast<size_t>(ue[j]) * a.n_up + uc[j]));
            g[j].x += p.x; g[j].y += p.y; g[j].z += p.z; g[j].w += p.w;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kAU; ++j) {
        if (ue[j] < 0) continue;
        const int e = ue[j], t = ut[j], c = uc[j];
        float hv[4];
        if (a.swiglu) {
          hv[0] = silu_fast(g[j].x) * u[j].x;
          hv[1] = silu_fast(g[j].y) * u[j].y;
          hv[2] = silu_fast(g[j].z) * u[j].z;
          hv[3] = silu_fast(g[j].w) * u[j].w;
        } else {
          const float* b = a.b1 + static_cast<size_t>(e) * f + c;
          hv[0] = fmaxf(g[j].x + b[0], 0.f);
          hv[1] = fmaxf(g[j].y + b[1], 0.f);
          hv[2] = fmaxf(g[j].z + b[2], 0.f);
          hv[3] = fmaxf(g[j].w + b[3], 0.f);
        }
        uint2 o;
        o.x = pack_bf16(hv[0], hv[1]);
        o.y = pack_bf16(hv[2], hv[3]);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.h) + (static_cast<size_t>(e) * n_pad + t) * f + c) = o;
      }
    }
    fence_proxy_async_global();  // H is read next by TMA (async proxy)
  }
  if (!PU.direct) grid_barrier(a.sched, ++nbar, s_abort, a.timeout_ns, a.status);

  // ---------------------------------------------------------------- phase D (+ combine per tile)
  if (warp == 0) {
    if (lane == 0) produce(PD, pre, pre_start);
  } else if (warp == 1) {
    if (lane == 0) mma(PD);
  } else {
    epilogue(PD, a.tile_combine != 0);
  }
  if (!a.tile_combine) {
    // ------------------------------------------------------------ phase C: combine after a barrier
    grid_barrier(a.sched, ++nbar, s_abort, a.timeout_ns, a.status);
    if (!*s_abort) {
      const int d = a.d, d4 = d / 4;
      const size_t rows_total = static_cast<size_t>(E) * d;
      for (int w = gtid; w < T * d4; w += gstride) {
        const int t = w / d4, c = (w - t * d4) * 4;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < Sl; ++k) {
          const int e = a.idx[t * Sl + k];
          const size_t grow = static_cast<size_t>(e) * d + c;
          float4 p[kDecodeSplitsDown];
#pragma unroll
          for (int sp = 0; sp < kDecodeSplitsDown; ++sp)
            p[sp] = sp < PD.S ? __ldcg(reinterpret_cast<const float4*>(
                                    a.partial + (static_cast<size_t>(sp) * n_pad + t) * rows_total + grow))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          float4 v = p[0];
#pragma unroll
          for (int sp = 1; sp < kDecodeSplitsDown; ++sp)
            if (sp < PD.S) {
              v.x += p[sp].x; v.y += p[sp].y; v.z += p[sp].z; v.w += p[sp].w;
            }
          if (a.b2) {
            const float* b = a.b2 + grow;
            v.x += b[0]; v.y += b[1]; v.z += b[2]; v.w += b[3];
          }
          const float gk = a.gate[t * Sl + k];
          const float y[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = k == 0 ? __fmul_rn(gk, y[i]) : __fadd_rn(o[i], __fmul_rn(gk, y[i]));
        }
        if (a.out_bf16) {
          uint2 pk;
          pk.x = pack_bf16(o[0], o[1]);
          pk.y = pack_bf16(o[2], o[3]);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(t) * d + c) = pk;
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<size_t>(t) * d + c) =
              make_float4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }

  // row bookkeeping of the dispatch layout (what get_routing reports; nothing here reads it)
  for (int i = gtid; i < n_slots; i += gstride) {
    const int t = i / Sl;
    const int r = a.chunk_base[static_cast<size_t>(t / kRouterChunk) * E + a.idx[i]] + a.row_of[i];
    if (r >= 0 && r < a.rows_alloc) {
      a.row_of[i] = r;
      a.token_of_row[r] = t;
    } else {
      atomicOr(a.status, kStatusBadRow);
    }
  }

  // ---------------------------------------------------------------- teardown
  if (warp == 0 && lane == 0) {
    // copies issued but never consumed (only after a timeout) land before the CTA leaves
    for (int s = 0; s < nst; ++s)
      if (armed & (1u << s)) {
        volatile int never = 0;
        mbar_wait(full0 + 8 * s, (armed_phase >> s) & 1u, &never, a.timeout_ns);
      }
  }
  if (warp == 1 && lane == 0) {
    umma_commit(drain);
    volatile int never = 0;
    mbar_wait(drain, 0, &never, a.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, FTMEM_COLS);
  }
}

}  // namespace

cudaError_t prepare_decode_fused() {
  return cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FSMEM_BYTES);
}

// CTAs of the cooperative decode kernel that can be resident at once (0 on error).
int decode_fused_max_ctas(int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, FNUM_THREADS, FSMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm * num_sms;
}

cudaError_t launch_decode_fused(const CUtensorMap& tmW13, const CUtensorMap& tmX, const CUtensorMap& tmW2,
                                const CUtensorMap& tmH, const CUtensorMap& tmW13h, const FusedDecodeArgs& a, int grid,
                                cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(FNUM_THREADS);
  cfg.dynamicSmemBytes = FSMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_fused_kernel, tmW13, tmX, tmW2, tmH, tmW13h, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace colibri
