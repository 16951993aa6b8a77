// Internal declarations shared by the host code and the kernels of the MoE layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace colibri {

constexpr int kMaxRouted = 16;       // routed experts per layer (upper bound)
constexpr int kMaxE = kMaxRouted + 1;  // scheduled experts: routed + the optional shared expert
constexpr int kMaxTopK = 4;
constexpr int kMaxSlots = kMaxTopK + 1;  // rows per token: its k routed experts + the shared expert
constexpr int kRowTile = 128;        // expert row segments start on multiples of this (GEMM M tile)
constexpr int kRouterChunk = 32;     // tokens per router CTA (4 per warp)
constexpr int kRouterThreads = 256;
constexpr int kRouterMaxSmem = 96 * 1024;  // W_r columns staged per router pass (dynamic smem)
constexpr int kDecodeMaxT = 128;           // most tokens of a decode-path batch (cooperative kernel)
constexpr int kDecodeSepMaxT = 64;         // most tokens of a batch on the separate decode kernels
constexpr int kDecodeSplitsUp = 2;         // most K splits of the decode up projection
constexpr int kDecodeSplitsDown = 8;       // most K splits of the decode down projection

// Device status word bits (sticky until read by colibri_moe_device_status).
enum : int32_t {
  kStatusTimeoutProducer = 1 << 0,
  kStatusTimeoutMma = 1 << 1,
  kStatusTimeoutEpilogue = 1 << 2,
  kStatusBadRow = 1 << 3,
  kStatusTimeoutGridSync = 1 << 4,
  kStatusTimeoutRouter = 1 << 5,
  kStatusWaitProbe = 1 << 6,  // the failure-detection probe's wait ran out (as it is meant to)
  kStatusTimeoutRouteSync = 1 << 7,  // the router's grid barrier (fused dispatch) gave up
};

// Routing summary in device memory.  Written by the last CTA of the router kernel, read by
// every later stage of the same forward.
constexpr int kRouterSplitMaxChunks = 32;  // the split router serves batches of up to 1024 tokens

struct Sched {
  int32_t counts[kMaxE];           // rows routed to each expert
  int32_t offsets[kMaxE + 1];      // first row of each expert segment (segments padded to 128 rows)
  int32_t mtile_start[kMaxE + 1];  // prefix sum of ceil(counts / 128): M tiles before each expert
  uint32_t ticket;                 // router CTAs finished (reset to 0 by the last one)
  uint32_t grid_sync;              // arrivals at the cooperative decode kernel's grid barriers (reset by the router)
  uint32_t tile_ctr[2];            // next tile of the up / down CTA-pair GEMM (reset by the router)
  uint32_t split_ticket[kRouterSplitMaxChunks];  // split router: CTAs done per chunk (self-resetting)
  int32_t status;                  // device status word (kStatus* bits)
  uint32_t wm_done[kMaxE];         // fused weight-major GEMM: up items' epilogue warps done per expert
  uint32_t wm_cleared;             // fused weight-major GEMM: warps done clearing out (both reset by the router)
};

// The GEMMs' run-time counters, cleared by the router of every forward (one thread).
__device__ __forceinline__ void reset_gemm_counters(Sched* s) {
  s->tile_ctr[0] = s->tile_ctr[1] = 0;
  for (int e = 0; e < kMaxE; ++e) s->wm_done[e] = 0;
  s->wm_cleared = 0;
}

struct RouterArgs {
  const void* x;           // [T, d] dtype
  const void* w_router;    // [E, d] dtype
  const float* b_router;   // [E] or nullptr
  int T, d, E;             // E = routed experts
  int dchunk;              // columns of W_r staged in shared memory per pass
  int32_t* idx;            // [T, S]
  float* gate;             // [T, S]
  int32_t* rank;           // [T, S] rank inside the router chunk; rewritten to the row by gather
  int32_t* hist;           // [nchunks, Ex] counts per chunk, rewritten to first row per (chunk, expert)
  Sched* sched;
  int k;                   // routed experts per token (1..4)
  int gate_mode;           // 0 softmax over the selected experts, 1 full softmax
  int shared;              // 1: slot k of every token is the shared expert (index E, gate 1)
  int S;                   // slots per token = k + shared
  int Ex;                  // scheduled experts = E + shared
  float* zero_out;         // fused combine: out [T, d] fp32 rows of this CTA's tokens cleared, else nullptr
  uint32_t* tile_done;     // cooperative decode kernel's per-tile counters, cleared by the last CTA
  int n_tile_done;
  float* split_part;       // split router: partial logits [chunks][splits][32][EMAX], or nullptr
  // Dispatch fused into the split router (bf16 prefill batches of 9..1024 tokens; cooperative launch,
  // every CTA resident): each CTA finds its chunk's rows from all chunks' histograms after a grid
  // barrier and writes Xp,
  // row_of, token_of_row and gate_of_row itself -- no last-CTA scan, no separate dispatch kernel.
  // `rank` then holds only the in-chunk ranks (a buffer of its own), row_of the rows.
  void* xp;                // [rows_alloc, d], or nullptr: dispatch not fused
  int32_t* row_of;         // [T, S]
  int32_t* token_of_row;   // [rows_alloc]
  float* gate_of_row;      // [rows_alloc] or nullptr
  int64_t rows_alloc;
  uint32_t* route_sync;    // grid barrier arrivals: zero at launch, cleared again by the up GEMM
  uint64_t timeout_ns;     // bound on the grid barrier
};

struct GatherArgs {
  const void* x;           // [T, d]
  const int32_t* idx;      // [T, S]
  int32_t* row_of;         // [T, S] in: rank in chunk, out: row
  const int32_t* chunk_base;  // [nchunks, Ex]
  int T, d, E;             // E = scheduled experts (Ex)
  int S;
  int64_t rows_alloc;
  void* xp;                // [rows_alloc, d], or nullptr: bookkeeping only (A gathered by the GEMM)
  int32_t* token_of_row;   // [rows_alloc]
  Sched* sched;
  const float* gate;       // [T, S]
  float* gate_of_row;      // [rows_alloc] or nullptr
};

struct CombineArgs {
  const float* y;          // [rows, d] fp32
  const int32_t* row_of;   // [T, S]
  const float* gate;       // [T, S]
  int T, d;
  void* out;               // [T, d] fp32 or bf16
  int S;
};

enum GemmEpilogue : int {
  kEpiSwiGLU = 0,    // up projection, gate/up interleaved -> H = silu(g) * u
  kEpiReluBias = 1,  // up projection -> H = max(acc + b1, 0)
  kEpiStoreF32 = 2,  // down projection -> Y = acc (+ b2)
  kEpiCombineF32 = 3,  // down projection fused with the combine: out[token] += gate * (acc (+ b2))
};

struct GemmArgs {
  const Sched* sched;
  int E;
  int K;                    // reduction length
  int n_per_expert;         // rows of the weight operand per expert
  int n_tiles;              // column tiles per expert
  void* out;                // H or Y
  int64_t ldo;              // elements per output row
  const float* bias;        // [E, out_cols] or nullptr
  int out_cols;             // output columns per expert (f for up, d for down)
  uint64_t timeout_ns;      // bound on every wait inside the kernel
  int32_t* status;          // device status word (Sched::status)
  const int32_t* token_of_row;  // kEpiCombineF32 and gathered A: token of each row
  const float* gate_of_row;     // kEpiCombineF32: gate of each row
  const void* gather_x;         // gathered A: token rows x [T, K] bf16 (16-byte aligned rows)
  uint32_t* tile_ctr;           // CTA-pair kernel: next tile index to hand out (cleared by the router)
  float4* zero_out;             // up GEMM with the combine fused downstream: out cleared by two extra
  int64_t zero_vec4;            //   warps per CTA (zero_vec4 float4s), else nullptr
  uint32_t* clear_word;         // up GEMM after a router with fused dispatch: its grid barrier counter,
                                //   set to zero by CTA 0 once the router has completed, else nullptr
  int half_tiles;               // CTA-pair kernel: an expert's odd last 128-row M tile runs as an M=128
                                //   pair tile (64 rows per CTA) instead of an M=256 tile half of padding
  const int32_t* row_map;       // CTA-pair kernel, kEpiStoreF32: output row of each A row, or nullptr
  int wm_ntok;                  // weight-major kernel: token rows per tile (a multiple of 32, <= 256)
};

// Weight-major CTA-pair GEMM (gemm_tcgen05_wm.cu): the weight operand's tensor map (128-row boxes, or
// 64-row boxes for the SwiGLU up projection's gate / up halves) and the token operand's (Xp or H) with
// boxes of 16, 32, ..., 128 rows: tok[i] loads 16 (i + 1) rows, half of a token tile of 32 (i + 1).
constexpr int kWmTokMaps = 8;
struct WmMaps {
  CUtensorMap w;
  CUtensorMap tok[kWmTokMaps];
};
// Both projections in one launch (launch_wm_fused): the up projection's items, then the down
// projection's; a down item of expert e starts once every up item of e has written its H rows.
struct WmFused {
  WmMaps maps[2];  // up, down
  GemmArgs args[2];
};

constexpr int kZeroWarp0 = 6;   // the clearing warps follow producer, MMA and the 4 epilogue warps
constexpr int kZeroWarps = 2;

// Clears this CTA's share of out[0 .. n4) (float4s) with streaming stores: the share of CTA c of g
// is [c*n4/g, (c+1)*n4/g).  Run by the kZeroWarps extra warps while the mainloop is tensor-bound,
// so the 4 bytes per output element cost no step time.
__device__ __forceinline__ void clear_share(float4* out, int64_t n4, int cta, int nctas, int tid) {
  const int64_t b = n4 * cta / nctas, e = n4 * (cta + 1) / nctas;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = b + tid; i < e; i += 32 * kZeroWarps) __stcs(out + i, z);
}

// Decode (weight-streaming) GEMM: P[s][tok][row] partial sums over K split s.
struct DecodeArgs {
  const Sched* sched;
  int E;
  int K;                    // reduction length
  int n_per_expert;         // weight rows per expert (multiple of 128)
  int n_pad;                // token columns (16, 32, 48 or 64), >= every expert's count
  int s_max;                // most K splits
  int grid_ref;             // CTA count the split choice is computed for (same in every kernel)
  float* partial;           // [s_max][n_pad][E * n_per_expert] fp32
  uint64_t timeout_ns;
  int32_t* status;
};

struct DecodeActArgs {
  const Sched* sched;
  int E, K, n_per_expert, n_pad, s_max, grid_ref;
  int f;                    // H columns
  const float* partial;
  const float* bias;        // b1 [E, f] (ReLU) or nullptr
  void* h;                  // H [rows, f] bf16
};

struct DecodeCombineArgs {
  const Sched* sched;
  int E, K, n_pad, s_max, grid_ref;
  int d, T;
  const float* partial;     // down-projection partials, rows = E * d
  const float* bias;        // b2 [E, d] or nullptr
  const int32_t* idx;       // [T, S]
  const int32_t* row_of;    // [T, S]
  const float* gate;        // [T, S]
  void* out;
  int S;
};

// Cooperative decode kernel (T <= 128): up projection, activation, down projection, combine.
struct FusedDecodeArgs {
  Sched* sched;
  int E;                    // scheduled experts (routed + shared)
  int d, f, n_up;           // model width, hidden width, up-projection weight rows per expert
  int T, n_pad, S;          // tokens, token columns (16..128, >= T), slots per token
  const int32_t* idx;       // [T, S] from the router
  const float* gate;        // [T, S]
  int32_t* row_of;          // [T, S] in: rank in chunk, out: row of the dispatch layout
  int32_t* token_of_row;    // [rows_alloc]
  const int32_t* chunk_base;  // [nchunks, E] first row of each (chunk, expert)
  int64_t rows_alloc;
  float* partial;           // [splits][n_pad][E * rows] fp32
  const float* b1;          // [E, f] (ReLU) or nullptr
  const float* b2;          // [E, d] or nullptr
  void* h;                  // H rows e * n_pad + t, bf16 [.., f]
  void* out;                // [T, d]
  int out_bf16, swiglu;
  uint64_t timeout_ns;
  int32_t* status;
  uint32_t* tile_done;      // [d / 128] items finished per down-projection weight tile (self-resetting)
  int tile_combine;         // 1: combine per tile by its last CTA; 0: after a grid barrier
  int direct_h;             // 1: an unsplit up projection writes H in its epilogue (no phase A)
};

// fp32 SIMT grouped GEMM operands (row-major, K contiguous)
struct SimtGemmArgs {
  const Sched* sched;
  int E, K, N;              // N = output columns per expert
  const float* a;           // [rows, K]
  const float* b;           // [E * N, K]  (W1 / W_gate / W2)
  const float* b3;          // [E * N, K]  W_up for SwiGLU, else nullptr
  const float* bias;        // [E, N] or nullptr
  float* out;               // [rows, N]
  // fused combine (store epilogue, two slots, fp32 out): comb_out[token_of_row[r]] += gate_of_row[r] * y[r]
  // onto rows the router cleared, instead of writing out
  const int* token_of_row = nullptr;
  const float* gate_of_row = nullptr;
  float* comb_out = nullptr;
};

// Expert parallelism (the experts split over several GPUs).
struct EpPackArgs {
  const void* x;            // [T, d]
  const int32_t* idx;       // [T, k]
  int32_t* row_of;          // [T, k] in: rank inside the router chunk, out: row of the send buffer
  const int32_t* chunk_base;  // [nchunks, E] first padded row of each (chunk, expert)
  const Sched* sched;       // the router's summary (counts, padded offsets)
  int T, d, E, k;
  void* send;               // [T * k, d]: rows grouped by expert, ascending token inside each
  int32_t* send_counts;     // [E] rows per expert
  int32_t* status;
};

// How the rows an expert rank receives (source-major blocks) map onto its padded expert segments.
struct EpPlan {
  int32_t n_seg;              // ep_size * El segments (<= kMaxRouted), source-major
  int32_t El;                 // local experts
  int32_t src[kMaxRouted];    // first received row of segment g = (source p, local expert j)
  int32_t dst[kMaxRouted];    // its first row in Xp: offsets[j] + rows of j from sources before p
  int32_t counts[kMaxE];      // rows per local expert
  int32_t offsets[kMaxE + 1]; // 128-row padded segment starts
  int32_t mstart[kMaxE + 1];  // M tiles before each local expert
};

struct EpRegroupArgs {
  const void* recv;         // [R, d] received rows
  void* xp;                 // Xp
  int R;
  int row_bytes;            // d * element size (a multiple of 16)
  Sched* sched;             // the expert role's schedule
  EpPlan plan;
  int32_t* recv_of_row;     // [rows of Xp] receive index of each row it fills, or nullptr
};

struct EpUnregroupArgs {
  const float* y;           // Y [rows, d] fp32 (padded layout)
  float* y_out;             // [R, d] fp32 in receive order
  int R, d;
  EpPlan plan;
};

// Programmatic dependent launch: a kernel launched with pdl_launch may start (and run its prologue)
// while the previous kernel on the stream drains; it must call pdl_wait() before touching anything
// an earlier kernel wrote (pdl_wait returns once every prerequisite grid has completed and its
// memory is visible; without the launch attribute it returns at once).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Decode-path helpers shared by the separate-kernel and the cooperative decode path.
// Number of K splits: the smallest S whose items fill >= 95 % of their waves, else the best fill (a
// wave 8 % short, as 1120 unsplit items on 152 CTAs, costs more than the split sums).
__device__ __forceinline__ int decode_splits(int items0, int kblocks, int grid, int s_max) {
  int best = 1;
  int best_num = -1, best_den = 1;
  for (int S = 1; S <= s_max && S <= kblocks; ++S) {
    const int items = items0 * S;
    const int waves = (items + grid - 1) / grid;
    if (items >= grid && items * 20 >= waves * grid * 19) return S;
    if (static_cast<long long>(items) * best_den > static_cast<long long>(best_num) * (waves * grid)) {
      best_num = items;
      best_den = waves * grid;
      best = S;
    }
  }
  return best;
}

__device__ __forceinline__ int active_experts(const Sched* sc, int E, int* list) {
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (sc->counts[e] > 0) list[n++] = e;
  return n;
}

// launchers (return cudaGetLastError() of the launch)
cudaError_t launch_router(int dtype, const RouterArgs& a, int nchunks, cudaStream_t s);
cudaError_t launch_router_tma(const CUtensorMap& tmx, const RouterArgs& a, int nchunks, cudaStream_t s);
int router_tma_cols();  // the TMA-staged router needs d to be a multiple of this
cudaError_t launch_router_split(const RouterArgs& a, int nchunks, cudaStream_t s);
// The split router with the dispatch fused (a.xp set): a cooperative launch; the most chunks whose
// CTAs are all resident at once on the current device (0 on error).
cudaError_t launch_router_split_fused(const RouterArgs& a, int nchunks, cudaStream_t s);
int router_split_fused_max_chunks(int E, int num_sms);
int router_split_factor();  // CTAs per chunk of the split router (d must be a multiple of 32 x this)
cudaError_t launch_gather(int dtype, const GatherArgs& a, cudaStream_t s);
cudaError_t launch_combine(int out_dtype, const CombineArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_tc_gemm(int epi, bool gather_a, const CUtensorMap& tmA, const CUtensorMap& tmB,
                           const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_simt_gemm(int epi, const SimtGemmArgs& a, int max_mtiles, cudaStream_t s);
int router_smem_bytes(int dtype, int E, int dchunk);
// One-time kernel attribute set-up (dynamic shared memory limits) for the current device.
cudaError_t prepare_router(int dtype, int E);
cudaError_t prepare_tc_gemm();
cudaError_t prepare_decode_gemm();
cudaError_t prepare_pair_gemm();
int pair_gemm_max_ctas();
cudaError_t prepare_wm_gemm();
cudaError_t launch_wm_gemm(int epi, const WmMaps& maps, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_wm_fused(int epi_up, int epi_dn, const WmFused& f, int grid, cudaStream_t s);
int wm_gemm_max_ctas();
cudaError_t launch_pair_gemm(int epi, bool gather_a, const CUtensorMap& tmA, const CUtensorMap& tmA64,
                             const CUtensorMap& tmB, const GemmArgs& a, int grid, cudaStream_t s);
cudaError_t launch_decode_gemm(const CUtensorMap& tmW, const CUtensorMap& tmX, const DecodeArgs& a, int grid,
                               cudaStream_t s);
cudaError_t launch_decode_act(bool swiglu, const DecodeActArgs& a, cudaStream_t s);
cudaError_t prepare_decode_fused();
int decode_fused_max_ctas(int num_sms);
cudaError_t launch_decode_fused(const CUtensorMap& tmW13, const CUtensorMap& tmX, const CUtensorMap& tmW2,
                                const CUtensorMap& tmH, const CUtensorMap& tmW13h, const FusedDecodeArgs& a, int grid,
                                cudaStream_t s);
cudaError_t launch_decode_combine(int out_dtype, const DecodeCombineArgs& a, cudaStream_t s);
cudaError_t launch_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t s);
cudaError_t launch_ep_pack(int dtype, const EpPackArgs& a, cudaStream_t s);
cudaError_t launch_ep_regroup(const EpRegroupArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_ep_unregroup(const EpUnregroupArgs& a, int num_sms, cudaStream_t s);
int tc_gemm_block_n();
int tc_gemm_threads();

}  // namespace colibri
