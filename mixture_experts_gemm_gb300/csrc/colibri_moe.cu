// Host side of the C ABI declared in include/colibri_moe.h: context, device weight arena,
// workspace, argument validation and the launch sequence of one forward.
//
// Allocation happens in create (workspace sized for max_tokens) and load_weights (weight arena);
// forward only enqueues kernels (hnwysp.cn/news/30485 2.1: buffers allocated once, none on the
// forward path; m.nxbn.cn/news/48047 3.1: the maximum batch is fixed at initialisation).
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "colibri_moe.h"
#include "moe_internal.cuh"

using namespace colibri;

namespace colibri {
// Programmatic dependent launch between the forward's kernels; COLIBRI_MOE_PDL=0 turns it off.
bool pdl_enabled() {
  static const bool on = [] {
    const char* s = std::getenv("COLIBRI_MOE_PDL");
    return !(s && s[0] == '0');
  }();
  return on;
}
}  // namespace colibri

constexpr int kHostSlots = 3;  // staging slots of the pipelined host-buffer forward

struct colibri_moe {
  colibri_moe_config_t cfg{};
  int device = 0;
  int num_sms = 0;
  int64_t rows_alloc = 0;   // rows of Xp / H / Y
  int nchunks_max = 0;      // router chunks at max_tokens
  int dchunk = 0;           // router: W_r columns per shared-memory pass
  size_t esize = 0;         // bytes per element of x and weights
  size_t out_esize = 0;
  int n_up = 0;             // weight rows per expert of the up projection (2f SwiGLU bf16, f otherwise)
  int k = 2;                // routed experts per token
  int S = 2;                // rows per token: k routed (+1 shared)
  int Ex = 0;               // scheduled experts: E routed (+1 shared, index E)

  // weight arena (one allocation, every block 256-byte aligned)
  void* warena = nullptr;
  size_t warena_bytes = 0;
  void* w_router = nullptr;
  float* b_router = nullptr;
  void* w13 = nullptr;  // bf16 SwiGLU: [E, 2f, d], gate/up interleaved in blocks of 128 rows; else W1 [E, f, d]
  void* w3 = nullptr;   // fp32 SwiGLU: W_up [E, f, d]
  void* w2 = nullptr;   // [E, d, f]
  float* b1 = nullptr;  // [E, f]
  float* b2 = nullptr;  // [E, d]
  bool loaded = false;

  // workspace (one allocation)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* xp = nullptr;
  void* h = nullptr;
  float* y = nullptr;
  int32_t* idx = nullptr;
  float* gate = nullptr;
  int32_t* row_of = nullptr;
  int32_t* tok_of_row = nullptr;
  float* gate_of_row = nullptr;
  int32_t* hist = nullptr;
  Sched* sched = nullptr;
  // host-buffer staging: slot 0 serves forward_host; forward_host_async takes the slots in turn,
  // with two copy streams and per-slot events.  Three slots: a call's copy in waits for the copy out
  // of the call three back, so copy in, forward and copy out of one call spread over three calls'
  // time and the copies run at the host link's rate (with two slots that chain set the pace).
  void* x_stage[kHostSlots] = {};
  void* out_stage[kHostSlots] = {};
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev_in[kHostSlots] = {}, ev_done[kHostSlots] = {}, ev_free[kHostSlots] = {};
  int slot = 0;

  CUtensorMap tm_xp{}, tm_h{}, tm_w13{}, tm_w2{};
  // decode path (T <= decode_max_t): 128-row weight boxes, token boxes of 16, 32, ..., 128 rows
  CUtensorMap tm_w13_dec{}, tm_w2_dec{}, tm_xp_dec[kDecodeMaxT / 16]{}, tm_h_dec[kDecodeMaxT / 16]{};
  CUtensorMap tm_w13_half{};  // 64-row boxes: the cooperative decode kernel's gate/up pairs
  float* partial = nullptr;  // decode partial sums [splits][n_pad][E * rows]
  uint32_t* tile_done = nullptr;  // cooperative decode kernel: items done per down-projection tile
  float* split_part = nullptr;    // split router: partial logits of small batches
  // dispatch fused into the router (bf16 prefill path): in-chunk ranks, grid barrier counter, and
  // the most chunks each router variant runs with every CTA resident (0: never fused)
  int32_t* rank_buf = nullptr;    // [max_tokens, S]
  uint32_t* route_sync = nullptr;
  int fused_split_chunks = 0;
  bool fused_dispatch = true;
  int decode_max_t = 0;
  bool pair_gemm = false;    // prefill GEMMs on CTA pairs (256x256 tiles)
  bool fuse_combine = true;  // two-slot fp32 layers: gate-weighted combine inside the down GEMM
  bool gather_a = false;     // bf16 prefill: up GEMM reads A rows from x through token_of_row
  bool dynamic_tiles = true; // CTA-pair GEMMs take tiles in index order from a shared counter
  bool half_tiles = true;    // CTA-pair GEMMs run an expert's odd last M tile as an M=128 pair tile
  int wm_env = -1;           // weight-major GEMMs: -1 by batch size (wm_tile_rows), 0 never, n: token tile n
  bool wm_fused = true;      // ... both projections in one launch (needs the in-order tile hand-out)
  int wm_ctas = 0;           // co-resident CTAs of the weight-major kernel
  int pair_ctas = 0;         // co-resident CTAs of the pair kernel (persistent grid size)
  bool decode_fused = true;  // decode batches: one cooperative kernel after the router
  bool direct_h = true;      // ... whose unsplit up projection writes H in its epilogue
  int fused_ctas = 0;        // its grid (one CTA per SM)
  // expert parallelism (colibri_moe_ep_create): the context routes over all E experts but holds the
  // weights of experts [ep_first, ep_first + n_arena) only
  int ep_size = 0;           // 0: an ordinary context
  int ep_rank = 0;
  int ep_first = 0;
  int n_arena = 0;           // experts in the weight arena: Ex, or the local experts of an EP context
  int64_t ep_max_rows = 0;   // most rows one ep_experts call may receive
  Sched* ep_sched = nullptr; // schedule of the local experts' GEMMs (ep_experts)
  int32_t last_T = -1;
  int32_t last_kernels = 0;  // kernels enqueued by the last forward
  int32_t last_gemm = COLIBRI_GEMM_NONE;  // its grouped-GEMM form
  std::vector<cudaEvent_t> events;
  uint64_t timeout_ns = 2000000000ull;
};

namespace {

constexpr int kNumStages = 5;  // router, gather, up GEMM, down GEMM, combine
constexpr int kBox64 = 64 / 16 - 1;  // tm_xp_dec / tm_h_dec entry with 64-row boxes (the pair GEMM's half tiles)
// Cooperative decode kernel: batches up to this size combine per tile (no third grid barrier);
// measured on GB300 at the Mixtral shape: T=1 2 us faster, T=4 even, T >= 16 slower.
constexpr int kTileCombineMaxT = 4;
constexpr int kRouterTmaMinT = 1024;  // batches from this size use the TMA-staged router
constexpr int kRouterSplitMinT = 8;    // batches above this size (up to 32 chunks: 1024 tokens) use the split router
// (GB300, Mixtral-shaped decode steps: T=32 router stage 23.2 -> 16.9 us split; with the warp-match
// tail, T=16 432.7 -> 429.1 us per step split, T=1 and T=4 the same either way)

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2D bf16 tensor [rows, inner] row-major; box = 64 (inner) x box_rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A pointer the kernels may read/write: device (or managed) memory on the context's device.
bool is_device_ptr(const void* p, int device) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.device == device;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const char *pa = static_cast<const char*>(a), *pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

int check_config(const colibri_moe_config_t* c) {
  if (!c) return COLIBRI_ERR_INVALID_ARG;
  if (c->num_experts < 2 || c->num_experts > COLIBRI_MAX_EXPERTS) return COLIBRI_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > COLIBRI_MAX_TOP_K || c->top_k > c->num_experts) return COLIBRI_ERR_INVALID_ARG;
  if ((c->gate_mode != COLIBRI_GATE_SOFTMAX_SELECTED && c->gate_mode != COLIBRI_GATE_SOFTMAX_ALL) ||
      (c->has_shared_expert != 0 && c->has_shared_expert != 1))
    return COLIBRI_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->d_ff <= 0 || c->max_tokens <= 0 || c->max_tokens > (1 << 24))
    return COLIBRI_ERR_INVALID_ARG;
  if ((c->dtype != COLIBRI_DTYPE_F32 && c->dtype != COLIBRI_DTYPE_BF16) ||
      (c->out_dtype != COLIBRI_DTYPE_F32 && c->out_dtype != COLIBRI_DTYPE_BF16) ||
      (c->act != COLIBRI_ACT_RELU_BIAS && c->act != COLIBRI_ACT_SWIGLU) ||
      (c->has_router_bias != 0 && c->has_router_bias != 1))
    return COLIBRI_ERR_INVALID_ARG;
  if (c->d_model % 8 || c->d_ff % 8) return COLIBRI_ERR_UNSUPPORTED;
  if (c->dtype == COLIBRI_DTYPE_BF16) {
    const int bn = tc_gemm_block_n();
    if (c->d_model % bn) return COLIBRI_ERR_UNSUPPORTED;
    if (c->act == COLIBRI_ACT_SWIGLU && c->d_ff % (bn / 2)) return COLIBRI_ERR_UNSUPPORTED;
    if (c->act == COLIBRI_ACT_RELU_BIAS && c->d_ff % bn) return COLIBRI_ERR_UNSUPPORTED;
  }
  return COLIBRI_OK;
}

// Layers with two slots and an fp32 output fuse the combine into the down GEMM (tcgen05 or SIMT)
// unless COLIBRI_MOE_FUSED_COMBINE=0.
bool env_fuse_combine() {
  const char* s = std::getenv("COLIBRI_MOE_FUSED_COMBINE");
  return !(s && s[0] == '0');
}

// COLIBRI_MOE_GATHER=fused: the prefill up GEMM gathers its A rows from x (no Xp).  Off by default:
// on GB300 at the Mixtral shape it measured 2-4 % slower than the TMA-fed GEMM over Xp.
bool env_gather_a() {
  const char* s = std::getenv("COLIBRI_MOE_GATHER");
  return s && std::strcmp(s, "fused") == 0;
}

// bf16 prefill batches of 9..1024 tokens run the dispatch inside the split router (no separate
// dispatch kernel) unless COLIBRI_MOE_DISPATCH=separate.
bool env_fused_dispatch() {
  const char* s = std::getenv("COLIBRI_MOE_DISPATCH");
  return !(s && std::strcmp(s, "separate") == 0);
}

// CTA-pair GEMMs compute an expert's odd last 128-row M tile as an M=128 pair tile (64 rows per
// CTA) unless COLIBRI_MOE_PAIR_HALF=0, which pads it to a 256-row pair tile.
bool env_half_tiles() {
  const char* s = std::getenv("COLIBRI_MOE_PAIR_HALF");
  return !(s && s[0] == '0');
}

// Weight-major GEMMs for batches with few rows per expert: COLIBRI_MOE_WM=0 never, =n (a multiple of
// 32 in [32, 256]) always with token tiles of n rows, unset: by batch size (wm_tile_rows).
int env_wm() {
  const char* s = std::getenv("COLIBRI_MOE_WM");
  if (!s) return -1;
  const int n = std::atoi(s);
  return (n >= 32 && n <= 256 && n % 32 == 0) ? n : 0;
}

// CTA-pair GEMMs hand out tiles in index order at run time unless COLIBRI_MOE_TILE_ORDER=static.
bool env_dynamic_tiles() {
  const char* s = std::getenv("COLIBRI_MOE_TILE_ORDER");
  return !(s && std::strcmp(s, "static") == 0);
}

// Prefill GEMMs run on CTA pairs (cta_group::2) unless COLIBRI_MOE_GEMM=1sm selects the single-CTA kernel.
bool env_pair_gemm() {
  const char* s = std::getenv("COLIBRI_MOE_GEMM");
  return !(s && std::strcmp(s, "1sm") == 0);
}

// Decode-sized batches run the cooperative fused kernel unless COLIBRI_MOE_DECODE_FUSED=0 selects
// the separate kernels (dispatch, GEMM, activation, GEMM, combine).
// The cooperative decode kernel's up projection, when unsplit, writes H in its epilogue (no
// activation phase, one grid barrier fewer) unless COLIBRI_MOE_DECODE_DIRECT_H=0.
bool env_direct_h() {
  const char* s = std::getenv("COLIBRI_MOE_DECODE_DIRECT_H");
  return !(s && s[0] == '0');
}

bool env_decode_fused() {
  const char* s = std::getenv("COLIBRI_MOE_DECODE_FUSED");
  return !(s && s[0] == '0');
}

// Batches of up to this many tokens take the decode path: 128 for experts of at least 2^25 weights
// per matrix (d_model x d_ff; at the Mixtral shape the cooperative kernel wins up to 128 tokens),
// else 64 (with smaller experts the grouped GEMMs catch up between 64 and 96 tokens).
// COLIBRI_MOE_DECODE_MAX_T overrides (0 .. kDecodeMaxT; 0 turns the decode path off).
// Decode-path limit: batches of up to this many tokens run the cooperative weight-streaming kernel.
// With the weight-major GEMM available its fused form is as fast from ~32 tokens on for experts of at
// least 2^25 weights per matrix and from ~16 for smaller ones (Mixtral shape: 427 vs 427 us at 32
// tokens, 430 vs 440 at 64, 434 vs 470 at 128; 1.3B class: 112 vs 116 at 48; skewed 16 experts:
// 55 vs 58 at 32); without it (single-CTA GEMMs) the cooperative kernel serves up to 128 / 64.
int env_decode_max_t(int64_t d, int64_t f, bool weight_major) {
  const char* s = std::getenv("COLIBRI_MOE_DECODE_MAX_T");
  if (s) {
    long v = std::strtol(s, nullptr, 10);
    if (v >= 0 && v <= kDecodeMaxT) return static_cast<int>(v);
  }
  const bool large = d * f >= (int64_t{1} << 25);
  if (weight_major) return large ? 32 : 16;
  return large ? kDecodeMaxT : kDecodeSepMaxT;
}

uint64_t env_timeout_ns() {
  const char* s = std::getenv("COLIBRI_MOE_WAIT_TIMEOUT_MS");
  if (s) {
    long v = std::strtol(s, nullptr, 10);
    if (v > 0) return static_cast<uint64_t>(v) * 1000000ull;
  }
  return 2000000000ull;
}

}  // namespace

extern "C" {

const char* colibri_moe_strerror(int code) {
  switch (code) {
    case COLIBRI_OK: return "ok";
    case COLIBRI_ERR_INVALID_ARG: return "invalid argument";
    case COLIBRI_ERR_OOM: return "device allocation failed";
    case COLIBRI_ERR_BAD_WEIGHTS: return "missing or unexpected weight tensor";
    case COLIBRI_ERR_CUDA: return "CUDA call failed";
    case COLIBRI_ERR_STATE: return "call out of order (weights not loaded, or no forward yet)";
    case COLIBRI_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case COLIBRI_ERR_DEVICE: return "a kernel reported a failure in the device status word";
    default: return "unknown status code";
  }
}

void colibri_moe_destroy(colibri_moe_t* ctx) {
  if (!ctx) return;
  {
    DeviceGuard g(ctx->device);
    if (ctx->h2d) cudaStreamSynchronize(ctx->h2d);
    if (ctx->d2h) cudaStreamSynchronize(ctx->d2h);
    for (int i = 0; i < kHostSlots; ++i) {
      if (ctx->ev_in[i]) cudaEventDestroy(ctx->ev_in[i]);
      if (ctx->ev_done[i]) cudaEventDestroy(ctx->ev_done[i]);
      if (ctx->ev_free[i]) cudaEventDestroy(ctx->ev_free[i]);
    }
    if (ctx->h2d) cudaStreamDestroy(ctx->h2d);
    if (ctx->d2h) cudaStreamDestroy(ctx->d2h);
    if (ctx->warena) cudaFree(ctx->warena);
    if (ctx->ws) cudaFree(ctx->ws);
  }
  delete ctx;
}

}  // extern "C"

// Ordinary context (ep_size == 0) or the context of rank ep_rank of an expert-parallel layer.
static int create_impl(const colibri_moe_config_t* cfg, int device, int ep_rank, int ep_size, int64_t ep_max_rows,
                       colibri_moe_t** out) {
  if (!out) return COLIBRI_ERR_INVALID_ARG;
  *out = nullptr;
  int rc = check_config(cfg);
  if (rc) return rc;
  if (ep_size > 0) {
    if (ep_size > cfg->num_experts || cfg->num_experts % ep_size || ep_rank < 0 || ep_rank >= ep_size ||
        ep_max_rows <= 0 || ep_max_rows > (int64_t{1} << 26))
      return COLIBRI_ERR_INVALID_ARG;
    if (cfg->has_shared_expert) return COLIBRI_ERR_UNSUPPORTED;
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  if (device < 0 || device >= ndev) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return COLIBRI_ERR_CUDA;
  if (major != 10 || minor != 3) return COLIBRI_ERR_UNSUPPORTED;  // built for sm_103a only

  colibri_moe_t* c = new (std::nothrow) colibri_moe_t();
  if (!c) return COLIBRI_ERR_OOM;
  c->cfg = *cfg;
  c->device = device;
  c->num_sms = sms;
  c->timeout_ns = env_timeout_ns();
  c->pair_gemm = env_pair_gemm() && (sms % 2 == 0);
  c->fuse_combine = env_fuse_combine();
  c->gather_a = env_gather_a();
  c->dynamic_tiles = env_dynamic_tiles();
  c->half_tiles = env_half_tiles();
  c->wm_env = env_wm();
  {
    const char* wf = std::getenv("COLIBRI_MOE_WM_FUSED");
    c->wm_fused = !(wf && wf[0] == '0');
  }
  const int64_t d = cfg->d_model, f = cfg->d_ff, E = cfg->num_experts, T = cfg->max_tokens;
  c->esize = cfg->dtype == COLIBRI_DTYPE_F32 ? 4 : 2;
  c->out_esize = cfg->out_dtype == COLIBRI_DTYPE_F32 ? 4 : 2;
  c->n_up = (cfg->dtype == COLIBRI_DTYPE_BF16 && cfg->act == COLIBRI_ACT_SWIGLU) ? 2 * cfg->d_ff : cfg->d_ff;
  c->k = cfg->top_k;
  c->S = cfg->top_k + cfg->has_shared_expert;
  c->Ex = static_cast<int>(E) + cfg->has_shared_expert;
  const int64_t S = c->S, Ex = c->Ex;
  c->ep_size = ep_size;
  c->ep_rank = ep_rank;
  c->n_arena = ep_size > 0 ? static_cast<int>(E / ep_size) : c->Ex;
  c->ep_first = ep_size > 0 ? ep_rank * c->n_arena : 0;
  c->ep_max_rows = ep_size > 0 ? ep_max_rows : 0;
  // Xp / H / Y rows: every slot of max_tokens tokens, or the rows an expert rank may receive, plus
  // up to 127 padding rows per expert segment
  const int64_t gemm_rows = ep_size > 0 ? ep_max_rows : S * T;
  const int64_t gemm_experts = ep_size > 0 ? c->n_arena : Ex;
  c->rows_alloc = ((gemm_rows + (kRowTile - 1) * gemm_experts) + kRowTile - 1) / kRowTile * kRowTile;
  c->nchunks_max = static_cast<int>((T + kRouterChunk - 1) / kRouterChunk);
  {
    // W_r columns staged per router pass: at most 96 KB of shared memory
    const int vec_span = 32 * (16 / static_cast<int>(c->esize));
    const int emax = E <= 4 ? 4 : (E <= 8 ? 8 : 16);
    int dc = kRouterMaxSmem / (emax * static_cast<int>(c->esize));
    dc = dc / vec_span * vec_span;
    c->dchunk = static_cast<int>(d) < dc ? static_cast<int>(d) : dc;
  }
  const size_t h_es = cfg->dtype == COLIBRI_DTYPE_BF16 ? 2 : 4;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t o_xp = carve(c->rows_alloc * d * c->esize);
  const size_t o_h = carve(c->rows_alloc * f * h_es);
  const size_t o_y = carve(c->rows_alloc * d * 4);
  const size_t o_idx = carve(S * T * 4);
  const size_t o_gate = carve(S * T * 4);
  const size_t o_row = carve(S * T * 4);
  const size_t o_tok = carve(c->rows_alloc * 4);
  const size_t o_gor = carve(c->rows_alloc * 4);
  const size_t o_hist = carve(static_cast<size_t>(c->nchunks_max) * Ex * 4);
  const size_t o_sched = carve(sizeof(Sched));
  const size_t o_ep_sched = ep_size > 0 ? carve(sizeof(Sched)) : 0;
  // decode partial sums: bf16 layers whose batches can be decode-sized (an expert rank always runs
  // the grouped GEMMs: its rows come from every source)
  c->decode_max_t = (cfg->dtype == COLIBRI_DTYPE_BF16 && ep_size == 0)
                        ? env_decode_max_t(d, f, c->pair_gemm && c->wm_env != 0)
                        : 0;
  if (c->decode_max_t > T) c->decode_max_t = static_cast<int>(T);
  const int64_t npad_max = (c->decode_max_t + 15) / 16 * 16;
  const int64_t part_floats = c->decode_max_t > 0
                                  ? std::max<int64_t>(kDecodeSplitsUp * npad_max * Ex * c->n_up,
                                                      kDecodeSplitsDown * npad_max * Ex * d)
                                  : 0;
  const size_t o_part = carve(part_floats * 4);
  const size_t o_tiles = carve((d / 128 + 1) * sizeof(uint32_t));
  const size_t o_rank = carve(S * T * 4);
  const size_t o_rsync = carve(sizeof(uint32_t));
  const size_t o_spart = carve(static_cast<size_t>(kRouterSplitMaxChunks) * router_split_factor() * kRouterChunk *
                               16 * sizeof(float));
  size_t o_xs[kHostSlots], o_os[kHostSlots];
  for (int i = 0; i < kHostSlots; ++i) {  // (an expert-parallel context has no host-buffer forward)
    o_xs[i] = carve(ep_size > 0 ? 0 : T * d * c->esize);
    o_os[i] = carve(ep_size > 0 ? 0 : T * d * c->out_esize);
  }
  c->ws_bytes = off;
  if (cudaMalloc(&c->ws, c->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return COLIBRI_ERR_OOM;
  }
  char* b = static_cast<char*>(c->ws);
  c->xp = b + o_xp;
  c->h = b + o_h;
  c->y = reinterpret_cast<float*>(b + o_y);
  c->idx = reinterpret_cast<int32_t*>(b + o_idx);
  c->gate = reinterpret_cast<float*>(b + o_gate);
  c->row_of = reinterpret_cast<int32_t*>(b + o_row);
  c->tok_of_row = reinterpret_cast<int32_t*>(b + o_tok);
  c->gate_of_row = reinterpret_cast<float*>(b + o_gor);
  c->hist = reinterpret_cast<int32_t*>(b + o_hist);
  c->sched = reinterpret_cast<Sched*>(b + o_sched);
  c->ep_sched = ep_size > 0 ? reinterpret_cast<Sched*>(b + o_ep_sched) : nullptr;
  c->partial = part_floats > 0 ? reinterpret_cast<float*>(b + o_part) : nullptr;
  c->tile_done = reinterpret_cast<uint32_t*>(b + o_tiles);
  c->rank_buf = reinterpret_cast<int32_t*>(b + o_rank);
  c->route_sync = reinterpret_cast<uint32_t*>(b + o_rsync);
  c->split_part = reinterpret_cast<float*>(b + o_spart);
  for (int i = 0; i < kHostSlots; ++i) {
    c->x_stage[i] = b + o_xs[i];
    c->out_stage[i] = b + o_os[i];
  }
  bool streams_ok = cudaStreamCreateWithFlags(&c->h2d, cudaStreamNonBlocking) == cudaSuccess &&
                    cudaStreamCreateWithFlags(&c->d2h, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; i < kHostSlots && streams_ok; ++i)
    streams_ok = cudaEventCreateWithFlags(&c->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&c->ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&c->ev_free[i], cudaEventDisableTiming) == cudaSuccess;
  if (!streams_ok) {
    cudaGetLastError();
    colibri_moe_destroy(c);
    return COLIBRI_ERR_CUDA;
  }
  if (cudaMemset(c->ws, 0, c->ws_bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    colibri_moe_destroy(c);
    return COLIBRI_ERR_CUDA;
  }
  if (prepare_router(cfg->dtype, cfg->num_experts) != cudaSuccess ||
      (cfg->dtype == COLIBRI_DTYPE_BF16 && (prepare_tc_gemm() != cudaSuccess || prepare_decode_gemm() != cudaSuccess ||
                                             prepare_pair_gemm() != cudaSuccess || prepare_wm_gemm() != cudaSuccess ||
                                             prepare_decode_fused() != cudaSuccess))) {
    cudaGetLastError();
    colibri_moe_destroy(c);
    return COLIBRI_ERR_CUDA;
  }
  if (c->pair_gemm) {
    c->pair_ctas = pair_gemm_max_ctas();
    c->wm_ctas = wm_gemm_max_ctas();
    if (c->pair_ctas < 2 || c->wm_ctas < 2) c->pair_gemm = false;
  }
  c->fused_dispatch = env_fused_dispatch() && cfg->dtype == COLIBRI_DTYPE_BF16 && ep_size == 0;
  if (c->fused_dispatch) {
    c->fused_split_chunks = router_split_fused_max_chunks(cfg->num_experts, sms);
  }
  c->decode_fused = env_decode_fused() && c->decode_max_t > 0;
  c->direct_h = env_direct_h();
  if (c->decode_fused) {
    const int co = decode_fused_max_ctas(sms);
    c->fused_ctas = co < sms ? co : sms;
    if (c->fused_ctas < 1) c->decode_fused = false;
  }
  if (cfg->dtype == COLIBRI_DTYPE_BF16) {
    bool ok = make_tmap(&c->tm_xp, c->xp, d, c->rows_alloc, kRowTile) &&
              make_tmap(&c->tm_h, c->h, f, c->rows_alloc, kRowTile);
    for (int i = 0; ok && i < kDecodeMaxT / 16; ++i)
      ok = make_tmap(&c->tm_xp_dec[i], c->xp, d, c->rows_alloc, 16 * (i + 1)) &&
           make_tmap(&c->tm_h_dec[i], c->h, f, c->rows_alloc, 16 * (i + 1));
    if (!ok) {
      colibri_moe_destroy(c);
      return COLIBRI_ERR_CUDA;
    }
  }
  *out = c;
  return COLIBRI_OK;
}

extern "C" {

int colibri_moe_create(const colibri_moe_config_t* cfg, int device, colibri_moe_t** out) {
  return create_impl(cfg, device, 0, 0, 0, out);
}

int colibri_moe_ep_create(const colibri_moe_config_t* cfg, int32_t ep_rank, int32_t ep_size, int32_t max_recv_rows,
                          int device, colibri_moe_t** out) {
  if (ep_size < 1) {
    if (out) *out = nullptr;
    return COLIBRI_ERR_INVALID_ARG;
  }
  return create_impl(cfg, device, ep_rank, ep_size, max_recv_rows, out);
}

int colibri_moe_load_weights(colibri_moe_t* ctx, const colibri_moe_weights_t* w, void* stream) {
  if (!ctx || !w) return COLIBRI_ERR_INVALID_ARG;
  const colibri_moe_config_t& c = ctx->cfg;
  const int E = c.num_experts, Ex = ctx->n_arena;  // experts held in the arena
  const int first = ctx->ep_first;                  // arena expert e is expert first + e
  const bool swiglu = c.act == COLIBRI_ACT_SWIGLU;
  const bool shared = c.has_shared_expert != 0;
  // presence checks: every tensor the activation needs, and none it does not use
  if (!w->w_router || !w->w1 || !w->w2) return COLIBRI_ERR_BAD_WEIGHTS;
  if ((c.has_router_bias != 0) != (w->b_router != nullptr)) return COLIBRI_ERR_BAD_WEIGHTS;
  if (swiglu && (!w->w3 || w->b1 || w->b2)) return COLIBRI_ERR_BAD_WEIGHTS;
  if (!swiglu && (w->w3 || !w->b1 || !w->b2)) return COLIBRI_ERR_BAD_WEIGHTS;
  for (int e = first; e < first + (ctx->ep_size > 0 ? Ex : E); ++e) {  // an expert rank reads its own only
    if (!w->w1[e] || !w->w2[e]) return COLIBRI_ERR_BAD_WEIGHTS;
    if (swiglu && !w->w3[e]) return COLIBRI_ERR_BAD_WEIGHTS;
    if (!swiglu && (!w->b1[e] || !w->b2[e])) return COLIBRI_ERR_BAD_WEIGHTS;
  }
  if (shared) {
    if (!w->ws1 || !w->ws2 || (swiglu && (!w->ws3 || w->bs1 || w->bs2)) || (!swiglu && (w->ws3 || !w->bs1 || !w->bs2)))
      return COLIBRI_ERR_BAD_WEIGHTS;
  } else if (w->ws1 || w->ws3 || w->ws2 || w->bs1 || w->bs2) {
    return COLIBRI_ERR_BAD_WEIGHTS;
  }
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t d = c.d_model, f = c.d_ff, es = ctx->esize;
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t o_wr = carve(E * d * es);
  const size_t o_br = carve(E * 4);
  const size_t o_w13 = carve(Ex * static_cast<size_t>(ctx->n_up) * d * es);
  const size_t o_w3 = (swiglu && c.dtype == COLIBRI_DTYPE_F32) ? carve(Ex * f * d * es) : 0;
  const size_t o_w2 = carve(Ex * d * f * es);
  const size_t o_b1 = carve(Ex * f * 4);
  const size_t o_b2 = carve(Ex * d * 4);
  if (ctx->warena && ctx->warena_bytes != off) {
    cudaFree(ctx->warena);
    ctx->warena = nullptr;
  }
  ctx->loaded = false;
  if (!ctx->warena) {
    if (cudaMalloc(&ctx->warena, off) != cudaSuccess) {
      cudaGetLastError();
      return COLIBRI_ERR_OOM;
    }
    ctx->warena_bytes = off;
  }
  char* b = static_cast<char*>(ctx->warena);
  ctx->w_router = b + o_wr;
  ctx->b_router = c.has_router_bias ? reinterpret_cast<float*>(b + o_br) : nullptr;
  ctx->w13 = b + o_w13;
  ctx->w3 = (swiglu && c.dtype == COLIBRI_DTYPE_F32) ? b + o_w3 : nullptr;
  ctx->w2 = b + o_w2;
  ctx->b1 = swiglu ? nullptr : reinterpret_cast<float*>(b + o_b1);
  ctx->b2 = swiglu ? nullptr : reinterpret_cast<float*>(b + o_b2);

  bool ok = cudaMemcpyAsync(ctx->w_router, w->w_router, E * d * es, cudaMemcpyDefault, s) == cudaSuccess;
  if (ok && ctx->b_router)
    ok = cudaMemcpyAsync(ctx->b_router, w->b_router, E * 4, cudaMemcpyDefault, s) == cudaSuccess;
  const size_t mat = f * d * es;  // bytes of one [f, d] matrix
  // arena expert e < E: routed expert e; e == E: the shared expert
  for (int e = 0; ok && e < Ex; ++e) {
    const bool sh = ctx->ep_size == 0 && e == E;
    const int src = first + e;
    const void* W1 = sh ? w->ws1 : w->w1[src];
    const void* W3 = sh ? w->ws3 : (swiglu ? w->w3[src] : nullptr);
    const void* W2 = sh ? w->ws2 : w->w2[src];
    const float* B1 = sh ? w->bs1 : (swiglu ? nullptr : w->b1[src]);
    const float* B2 = sh ? w->bs2 : (swiglu ? nullptr : w->b2[src]);
    char* w13e = static_cast<char*>(ctx->w13) + static_cast<size_t>(e) * ctx->n_up * d * es;
    if (swiglu && c.dtype == COLIBRI_DTYPE_BF16) {
      // gate rows [128j, 128j+128) -> arena rows [256j, 256j+128); up rows -> [256j+128, 256j+256)
      const size_t blk = 128 * d * es;
      ok = cudaMemcpy2DAsync(w13e, 2 * blk, W1, blk, blk, f / 128, cudaMemcpyDefault, s) == cudaSuccess &&
           cudaMemcpy2DAsync(w13e + blk, 2 * blk, W3, blk, blk, f / 128, cudaMemcpyDefault, s) == cudaSuccess;
    } else {
      ok = cudaMemcpyAsync(w13e, W1, mat, cudaMemcpyDefault, s) == cudaSuccess;
      if (ok && ctx->w3)
        ok = cudaMemcpyAsync(static_cast<char*>(ctx->w3) + e * mat, W3, mat, cudaMemcpyDefault, s) == cudaSuccess;
    }
    if (ok) ok = cudaMemcpyAsync(static_cast<char*>(ctx->w2) + e * mat, W2, mat, cudaMemcpyDefault, s) == cudaSuccess;
    if (ok && !swiglu)
      ok = cudaMemcpyAsync(ctx->b1 + e * f, B1, f * 4, cudaMemcpyDefault, s) == cudaSuccess &&
           cudaMemcpyAsync(ctx->b2 + e * d, B2, d * 4, cudaMemcpyDefault, s) == cudaSuccess;
  }
  if (ok) ok = cudaStreamSynchronize(s) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  if (c.dtype == COLIBRI_DTYPE_BF16) {
    const int bn = tc_gemm_block_n();
    if (!make_tmap(&ctx->tm_w13, ctx->w13, d, static_cast<uint64_t>(Ex) * ctx->n_up, bn) ||
        !make_tmap(&ctx->tm_w2, ctx->w2, f, static_cast<uint64_t>(Ex) * d, bn) ||
        !make_tmap(&ctx->tm_w13_dec, ctx->w13, d, static_cast<uint64_t>(Ex) * ctx->n_up, kRowTile) ||
        !make_tmap(&ctx->tm_w2_dec, ctx->w2, f, static_cast<uint64_t>(Ex) * d, kRowTile) ||
        !make_tmap(&ctx->tm_w13_half, ctx->w13, d, static_cast<uint64_t>(Ex) * ctx->n_up, kRowTile / 2))
      return COLIBRI_ERR_CUDA;
  }
  ctx->loaded = true;
  return COLIBRI_OK;
}

// The router variant for this batch.  Large bf16 batches stream x into the router through shared
// memory by TMA (a per-call map of the caller's buffer); small ones read it straight from global
// memory.
enum RouterKind { kRouterSplit, kRouterTma, kRouterPlain };

static RouterKind router_kind(const colibri_moe_t* ctx, int32_t T, int nchunks) {
  const bool bf16 = ctx->cfg.dtype == COLIBRI_DTYPE_BF16;
  const int d = ctx->cfg.d_model;
  // 9..1024 tokens: the hidden dimension split over several CTAs per chunk (fewer tokens gain
  // nothing from it: one CTA's loads already take one or two rounds; more fill the GPU anyway)
  if (bf16 && T > kRouterSplitMinT && nchunks <= kRouterSplitMaxChunks && d % (32 * router_split_factor()) == 0)
    return kRouterSplit;
  if (bf16 && T >= kRouterTmaMinT && d % router_tma_cols() == 0) return kRouterTma;
  return kRouterPlain;
}

// Whether this batch's router runs the dispatch itself: the split router (9..1024 tokens) with every
// CTA of its grid resident at once.  (Larger batches keep the separate dispatch kernel: measured on
// GB300, its thousands of warps copy the rows faster than one router CTA per chunk after the
// barrier -- Mixtral prefill router + dispatch 59 -> 68 us, skewed 16-expert layer no gain -- while
// at 512 tokens the fused form saves the launch and the last-CTA scan: 1.3B-class step 130.7 -> 128.5 us.)
static bool can_fuse_dispatch(const colibri_moe_t* ctx, RouterKind kind, int nchunks) {
  return ctx->fused_dispatch && kind == kRouterSplit && nchunks <= ctx->fused_split_chunks;
}

static int enqueue_router(const colibri_moe_t* ctx, const RouterArgs& ra, const void* x, int32_t T, int nchunks,
                          cudaStream_t s) {
  const colibri_moe_config_t& c = ctx->cfg;
  const int d = c.d_model;
  const RouterKind kind = router_kind(ctx, T, nchunks);
  const bool fused = ra.xp != nullptr;  // the caller checked can_fuse_dispatch
  CUtensorMap tm_xr;
  if (kind == kRouterSplit) {
    if ((fused ? launch_router_split_fused(ra, nchunks, s) : launch_router_split(ra, nchunks, s)) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
  } else if (fused) {
    return COLIBRI_ERR_CUDA;  // (never: can_fuse_dispatch admits the split router only)
  } else if (kind == kRouterTma && make_tmap(&tm_xr, x, d, static_cast<uint64_t>(T), kRouterChunk)) {
    if (launch_router_tma(tm_xr, ra, nchunks, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  } else {
    if (launch_router(c.dtype, ra, nchunks, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  }
  return COLIBRI_OK;
}

// Token tile of the weight-major GEMMs for a prefill batch of T tokens, or 0 for the CTA-pair kernel.
// With about 256 rows or fewer per routed expert the CTA-pair kernel pads every expert to 256-row
// tiles and half of each ring stage holds token rows; the weight-major kernel sizes its token tiles
// to the rows (a quarter over the mean, rounded up to 32, so that most experts fit one tile) and
// keeps more weights in flight.  With more rows it keeps 256-row token tiles and is only ahead in its
// fused form (both projections in one launch) when the up projection is a few waves of items: then
// the last wave, which the separate launches leave part-empty, fills with down items (skewed 16
// experts, T=4096: 166 -> 158 us).  With many waves the CTA-pair kernel is ahead (1.3B-class T=2048:
// 216 vs 224 us, Mixtral-shaped T=3000: 1.32 vs 1.36 ms).
constexpr int64_t kWmMaxRowsSized = 256;  // rows per expert up to which token tiles follow the rows
constexpr int64_t kWmMaxWaves = 8;        // up-projection waves up to which the fused form is used
// rows: mean rows per routed expert; total_rows: rows over all scheduled experts (n_sched of them)
static int wm_tile_rows_for(const colibri_moe_t* ctx, int64_t rows, int64_t total_rows, int64_t n_sched) {
  if (ctx->wm_env >= 0) return ctx->wm_env;
  if (rows <= kWmMaxRowsSized) {
    int64_t nt = (rows + rows / 4 + 31) / 32 * 32;
    if (nt < 64) nt = 64;
    if (nt > 256) nt = 256;
    return static_cast<int>(nt);
  }
  if (!ctx->wm_fused || !ctx->dynamic_tiles) return 0;
  const int64_t items = (ctx->n_up / 256) * (total_rows / 256 + n_sched / 2);
  return items <= kWmMaxWaves * (ctx->wm_ctas / 2) ? 256 : 0;
}
static int wm_tile_rows(const colibri_moe_t* ctx, int32_t T) {
  return wm_tile_rows_for(ctx, static_cast<int64_t>(ctx->k) * T / ctx->cfg.num_experts,
                          ctx->S * static_cast<int64_t>(T), ctx->Ex);
}

static int enqueue_forward(colibri_moe_t* ctx, const void* x, void* out, int32_t T, cudaStream_t s) {
  const colibri_moe_config_t& c = ctx->cfg;
  const int E = ctx->Ex, d = c.d_model, f = c.d_ff;  // scheduled experts (routed + shared)
  const bool bf16 = c.dtype == COLIBRI_DTYPE_BF16;
  const bool swiglu = c.act == COLIBRI_ACT_SWIGLU;
  const bool timed = static_cast<int>(ctx->events.size()) == kNumStages + 1;
  auto mark = [&](int i) {
    if (timed && ctx->events[i]) cudaEventRecord(ctx->events[i], s);
  };
  const int nchunks = (T + kRouterChunk - 1) / kRouterChunk;
  int64_t max_mtiles = (ctx->S * static_cast<int64_t>(T) + (kRowTile - 1) * E) / kRowTile;
  if (max_mtiles > ctx->rows_alloc / kRowTile) max_mtiles = ctx->rows_alloc / kRowTile;

  // Two slots with an fp32 output on the prefill path: the down GEMM adds g * y straight into out
  // (cleared first); two fp32 additions onto zero give the same value in either order.
  // (the separate decode kernels serve up to kDecodeSepMaxT tokens, the cooperative kernel more)
  const bool decode = bf16 && T <= ctx->decode_max_t && (ctx->decode_fused || T <= kDecodeSepMaxT);
  const bool fuse = !decode && ctx->fuse_combine && ctx->S == 2 && c.out_dtype == COLIBRI_DTYPE_F32;
  // bf16 prefill: the up GEMM gathers its A rows from x through token_of_row instead of reading a
  // materialised Xp; the dispatch kernel then only writes the row bookkeeping.
  const bool gather_a = bf16 && !decode && ctx->gather_a;
  // decode batches: one cooperative kernel after the router, with x as the token operand of its up
  // GEMM (a tensor map of the caller's buffer, encoded per call)
  CUtensorMap tm_xt;
  const bool fused_decode = decode && ctx->decode_fused &&
                            make_tmap(&tm_xt, x, d, static_cast<uint64_t>(T), static_cast<uint32_t>((T + 15) / 16 * 16));
  mark(0);
  // With the combine fused, out is cleared before the down GEMM adds into it: by extra warps of the
  // (tensor-bound) up GEMM, or by the router on the gathered-A path whose extra warps gather and on
  // the fp32 (SIMT) path.
  float4* const clear_in_gemm = fuse && !gather_a ? static_cast<float4*>(out) : nullptr;
  const int64_t out_vec4 = static_cast<int64_t>(T) * d / 4;
  // bf16 prefill batches of 9..1024 tokens: the split router writes the dispatch (Xp rows and row
  // bookkeeping) itself; no dispatch kernel then runs
  const bool fused_disp = bf16 && !decode && !gather_a && can_fuse_dispatch(ctx, router_kind(ctx, T, nchunks), nchunks);
  RouterArgs ra{x, ctx->w_router, ctx->b_router, T, d, c.num_experts, ctx->dchunk, ctx->idx, ctx->gate,
                fused_disp ? ctx->rank_buf : ctx->row_of, ctx->hist, ctx->sched, ctx->k, c.gate_mode,
                c.has_shared_expert, ctx->S, ctx->Ex,
                fuse && (gather_a || !bf16) ? static_cast<float*>(out) : nullptr, ctx->tile_done, d / 128,
                ctx->split_part};
  if (fused_disp) {
    ra.xp = ctx->xp;
    ra.row_of = ctx->row_of;
    ra.token_of_row = ctx->tok_of_row;
    ra.gate_of_row = fuse ? ctx->gate_of_row : nullptr;
    ra.rows_alloc = ctx->rows_alloc;
    ra.route_sync = ctx->route_sync;
    ra.timeout_ns = ctx->timeout_ns;
  }
  const int rrc = enqueue_router(ctx, ra, x, T, nchunks, s);
  if (rrc) return rrc;
  mark(1);
  GatherArgs ga{x, ctx->idx, ctx->row_of, ctx->hist, T, d, E, ctx->S, ctx->rows_alloc,
                gather_a ? nullptr : ctx->xp, ctx->tok_of_row, ctx->sched, ctx->gate,
                fuse ? ctx->gate_of_row : nullptr};
  if (fused_decode) {
    // decode-sized batch, one cooperative kernel: up GEMM, activation, down GEMM, combine (it also
    // writes the dispatch bookkeeping, so no gather kernel runs)
    const int n_pad = (T + 15) / 16 * 16;
    mark(2);
    FusedDecodeArgs fa{ctx->sched, E, d, f, ctx->n_up, T, n_pad, ctx->S, ctx->idx, ctx->gate, ctx->row_of,
                       ctx->tok_of_row, ctx->hist, ctx->rows_alloc, ctx->partial, ctx->b1, ctx->b2, ctx->h, out,
                       c.out_dtype == COLIBRI_DTYPE_BF16 ? 1 : 0, swiglu ? 1 : 0, ctx->timeout_ns,
                       &ctx->sched->status, ctx->tile_done, T <= kTileCombineMaxT ? 1 : 0, ctx->direct_h ? 1 : 0};
    if (launch_decode_fused(ctx->tm_w13_dec, tm_xt, ctx->tm_w2_dec, ctx->tm_h_dec[n_pad / 16 - 1], ctx->tm_w13_half, fa,
                            ctx->fused_ctas, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    mark(3);
    mark(4);
    mark(5);
    ctx->last_T = T;
    ctx->last_kernels = 2;
    ctx->last_gemm = COLIBRI_GEMM_DECODE_FUSED;
    return COLIBRI_OK;
  }
  if (!fused_disp && launch_gather(c.dtype, ga, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  mark(2);
  if (decode) {
    // decode-sized batch: weight-streaming GEMMs with K splits, deterministic reductions
    const int n_pad = (T + 15) / 16 * 16;
    const int mi = n_pad / 16 - 1;
    DecodeArgs up{ctx->sched, E, d, ctx->n_up, n_pad, kDecodeSplitsUp, ctx->num_sms, ctx->partial,
                  ctx->timeout_ns, &ctx->sched->status};
    if (launch_decode_gemm(ctx->tm_w13_dec, ctx->tm_xp_dec[mi], up, ctx->num_sms, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    DecodeActArgs act{ctx->sched, E, d, ctx->n_up, n_pad, kDecodeSplitsUp, ctx->num_sms, f, ctx->partial, ctx->b1,
                      ctx->h};
    if (launch_decode_act(swiglu, act, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
    mark(3);
    DecodeArgs dn{ctx->sched, E, f, d, n_pad, kDecodeSplitsDown, ctx->num_sms, ctx->partial, ctx->timeout_ns,
                  &ctx->sched->status};
    if (launch_decode_gemm(ctx->tm_w2_dec, ctx->tm_h_dec[mi], dn, ctx->num_sms, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    mark(4);
    DecodeCombineArgs cb{ctx->sched, E, f, n_pad, kDecodeSplitsDown, ctx->num_sms, d, T, ctx->partial, ctx->b2,
                         ctx->idx, ctx->row_of, ctx->gate, out, ctx->S};
    if (launch_decode_combine(c.out_dtype, cb, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
    mark(5);
    ctx->last_T = T;
    ctx->last_kernels = 6;
    ctx->last_gemm = COLIBRI_GEMM_DECODE_SPLIT;
    return COLIBRI_OK;
  }
  const int wm_nt = bf16 && ctx->pair_gemm && !gather_a ? wm_tile_rows(ctx, T) : 0;
  const bool wm_one = wm_nt > 0 && ctx->wm_fused && ctx->dynamic_tiles;  // both projections in one launch
  if (wm_nt > 0) {
    // weight-major CTA pairs: 256 weight rows x a token tile of at most wm_nt rows per item
    const int64_t tok_tiles = ctx->S * static_cast<int64_t>(T) / wm_nt + E;
    WmMaps mu, md;
    mu.w = swiglu ? ctx->tm_w13_half : ctx->tm_w13_dec;
    md.w = ctx->tm_w2_dec;
    for (int i = 0; i < kWmTokMaps; ++i) {
      mu.tok[i] = ctx->tm_xp_dec[i];
      md.tok[i] = ctx->tm_h_dec[i];
    }
    GemmArgs up{ctx->sched, E, d, ctx->n_up, 0, ctx->h, f, ctx->b1, f, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, nullptr, nullptr,
                ctx->dynamic_tiles ? &ctx->sched->tile_ctr[0] : nullptr, clear_in_gemm, out_vec4,
                fused_disp ? ctx->route_sync : nullptr, 0};
    up.wm_ntok = wm_nt;
    GemmArgs dn{ctx->sched, E, f, d, 0, fuse ? out : ctx->y, d, ctx->b2, d, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, ctx->gate_of_row, nullptr,
                ctx->dynamic_tiles ? &ctx->sched->tile_ctr[1] : nullptr, nullptr, 0, nullptr, 0};
    dn.wm_ntok = wm_nt;
    const int64_t ctas_up = 2 * (ctx->n_up / 256) * tok_tiles, ctas_dn = 2 * (d / 256) * tok_tiles;
    const int epi_up = swiglu ? kEpiSwiGLU : kEpiReluBias, epi_dn = fuse ? kEpiCombineF32 : kEpiStoreF32;
    if (wm_one) {
      // one launch: a pair that runs out of up items goes on with down items of finished experts
      WmFused fz;
      fz.maps[0] = mu;
      fz.maps[1] = md;
      fz.args[0] = up;
      fz.args[1] = dn;
      const int64_t ctas = ctas_up + ctas_dn;
      const int grid = static_cast<int>(ctas < ctx->wm_ctas ? ctas : ctx->wm_ctas);
      if (launch_wm_fused(epi_up, epi_dn, fz, grid, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
      mark(3);
    } else {
      int grid = static_cast<int>(ctas_up < ctx->wm_ctas ? ctas_up : ctx->wm_ctas);
      if (launch_wm_gemm(epi_up, mu, up, grid, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
      mark(3);
      grid = static_cast<int>(ctas_dn < ctx->wm_ctas ? ctas_dn : ctx->wm_ctas);
      if (launch_wm_gemm(epi_dn, md, dn, grid, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
    }
  } else if (bf16 && ctx->pair_gemm) {
    // CTA pairs: 256-row tiles made of two 128-row tiles of one expert sharing the weight tile
    const int bn = tc_gemm_block_n();
    const int64_t max_pairs = (max_mtiles + E + 1) / 2;
    GemmArgs up{ctx->sched, E, d, ctx->n_up, ctx->n_up / bn, ctx->h, f, ctx->b1, f, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, nullptr, x,
                ctx->dynamic_tiles ? &ctx->sched->tile_ctr[0] : nullptr, clear_in_gemm, out_vec4,
                fused_disp ? ctx->route_sync : nullptr, ctx->half_tiles ? 1 : 0};
    int64_t ctas = 2 * max_pairs * up.n_tiles;
    int grid = static_cast<int>(ctas < ctx->pair_ctas ? ctas : ctx->pair_ctas);
    if (launch_pair_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, gather_a, ctx->tm_xp, ctx->tm_xp_dec[kBox64], ctx->tm_w13_dec, up,
                         grid, s) !=
        cudaSuccess)
      return COLIBRI_ERR_CUDA;
    mark(3);
    GemmArgs dn{ctx->sched, E, f, d, d / bn, fuse ? out : ctx->y, d, ctx->b2, d, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, ctx->gate_of_row, nullptr,
                ctx->dynamic_tiles ? &ctx->sched->tile_ctr[1] : nullptr, nullptr, 0, nullptr, ctx->half_tiles ? 1 : 0};
    ctas = 2 * max_pairs * dn.n_tiles;
    grid = static_cast<int>(ctas < ctx->pair_ctas ? ctas : ctx->pair_ctas);
    if (launch_pair_gemm(fuse ? kEpiCombineF32 : kEpiStoreF32, false, ctx->tm_h, ctx->tm_h_dec[kBox64], ctx->tm_w2_dec, dn, grid,
                         s) !=
        cudaSuccess)
      return COLIBRI_ERR_CUDA;
  } else if (bf16) {
    const int bn = tc_gemm_block_n();
    GemmArgs up{ctx->sched, E, d, ctx->n_up, ctx->n_up / bn, ctx->h, f, ctx->b1, f, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, nullptr, x, nullptr, clear_in_gemm, out_vec4,
                fused_disp ? ctx->route_sync : nullptr};
    int64_t tiles = max_mtiles * up.n_tiles;
    int grid = static_cast<int>(tiles < ctx->num_sms ? tiles : ctx->num_sms);
    if (launch_tc_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, gather_a, ctx->tm_xp, ctx->tm_w13, up, grid, s) !=
        cudaSuccess)
      return COLIBRI_ERR_CUDA;
    mark(3);
    GemmArgs dn{ctx->sched, E, f, d, d / bn, fuse ? out : ctx->y, d, ctx->b2, d, ctx->timeout_ns,
                &ctx->sched->status, ctx->tok_of_row, ctx->gate_of_row};
    tiles = max_mtiles * dn.n_tiles;
    grid = static_cast<int>(tiles < ctx->num_sms ? tiles : ctx->num_sms);
    if (launch_tc_gemm(fuse ? kEpiCombineF32 : kEpiStoreF32, false, ctx->tm_h, ctx->tm_w2, dn, grid, s) !=
        cudaSuccess)
      return COLIBRI_ERR_CUDA;
  } else {
    SimtGemmArgs up{ctx->sched, E, d, f, static_cast<const float*>(ctx->xp), static_cast<const float*>(ctx->w13),
                    static_cast<const float*>(ctx->w3), ctx->b1, static_cast<float*>(ctx->h)};
    if (launch_simt_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, up, static_cast<int>(max_mtiles), s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    mark(3);
    SimtGemmArgs dn{ctx->sched, E, f, d, static_cast<const float*>(ctx->h), static_cast<const float*>(ctx->w2),
                    nullptr, ctx->b2, ctx->y, ctx->tok_of_row, ctx->gate_of_row, fuse ? static_cast<float*>(out) : nullptr};
    if (launch_simt_gemm(kEpiStoreF32, dn, static_cast<int>(max_mtiles), s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  }
  mark(4);
  if (!fuse) {
    CombineArgs ca{ctx->y, ctx->row_of, ctx->gate, T, d, out, ctx->S};
    if (launch_combine(c.out_dtype, ca, ctx->num_sms, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  }
  mark(5);
  ctx->last_T = T;
  ctx->last_kernels = (fuse ? 4 : 5) - (fused_disp ? 1 : 0) - (wm_one ? 1 : 0);
  ctx->last_gemm = wm_one ? COLIBRI_GEMM_WEIGHT_MAJOR_FUSED
                   : wm_nt > 0 ? COLIBRI_GEMM_WEIGHT_MAJOR
                   : !bf16 ? COLIBRI_GEMM_SIMT
                   : ctx->pair_gemm ? COLIBRI_GEMM_PAIR : COLIBRI_GEMM_SINGLE_CTA;
  return COLIBRI_OK;
}

int colibri_moe_forward(colibri_moe_t* ctx, const void* x, void* out, int32_t T, void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size > 0) return COLIBRI_ERR_UNSUPPORTED;  // an expert rank: ep_dispatch / ep_experts / ep_combine
  if (T < 0 || T > ctx->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
  if (!ctx->loaded) return COLIBRI_ERR_STATE;
  if (T == 0) {
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!x || !out) return COLIBRI_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->esize;
  const size_t ob = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->out_esize;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15) return COLIBRI_ERR_INVALID_ARG;
  if (overlap(x, xb, out, ob)) return COLIBRI_ERR_INVALID_ARG;
  if (!is_device_ptr(x, ctx->device) || !is_device_ptr(out, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  return enqueue_forward(ctx, x, out, T, static_cast<cudaStream_t>(stream));
}

int colibri_moe_forward_host(colibri_moe_t* ctx, const void* x_host, void* out_host, int32_t T, void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size > 0) return COLIBRI_ERR_UNSUPPORTED;  // an expert rank: ep_dispatch / ep_experts / ep_combine
  if (T < 0 || T > ctx->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
  if (!ctx->loaded) return COLIBRI_ERR_STATE;
  if (T == 0) {
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!x_host || !out_host) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->esize;
  const size_t ob = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->out_esize;
  // after any pipelined call still copying out of the staging slots
  for (int i = 0; i < kHostSlots; ++i)
    if (cudaStreamWaitEvent(s, ctx->ev_free[i], 0) != cudaSuccess) {
      cudaGetLastError();
      return COLIBRI_ERR_CUDA;
    }
  if (cudaMemcpyAsync(ctx->x_stage[0], x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  int rc = enqueue_forward(ctx, ctx->x_stage[0], ctx->out_stage[0], T, s);
  if (rc) return rc;
  if (cudaMemcpyAsync(out_host, ctx->out_stage[0], ob, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  return COLIBRI_OK;
}

int colibri_moe_forward_host_async(colibri_moe_t* ctx, const void* x_host, void* out_host, int32_t T,
                                   void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size > 0) return COLIBRI_ERR_UNSUPPORTED;
  if (T < 0 || T > ctx->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
  if (!ctx->loaded) return COLIBRI_ERR_STATE;
  if (T == 0) {
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!x_host || !out_host) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int k = ctx->slot;
  void* xs = ctx->x_stage[k];
  void* os = ctx->out_stage[k];
  const size_t xb = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->esize;
  const size_t ob = static_cast<size_t>(T) * ctx->cfg.d_model * ctx->out_esize;
  // slot k is free once the call kHostSlots back has copied its result out (its forward read x before)
  if (cudaStreamWaitEvent(ctx->h2d, ctx->ev_free[k], 0) != cudaSuccess ||
      cudaMemcpyAsync(xs, x_host, xb, cudaMemcpyHostToDevice, ctx->h2d) != cudaSuccess ||
      cudaEventRecord(ctx->ev_in[k], ctx->h2d) != cudaSuccess || cudaStreamWaitEvent(s, ctx->ev_in[k], 0) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  const int rc = enqueue_forward(ctx, xs, os, T, s);
  if (rc) return rc;
  if (cudaEventRecord(ctx->ev_done[k], s) != cudaSuccess || cudaStreamWaitEvent(ctx->d2h, ctx->ev_done[k], 0) != cudaSuccess ||
      cudaMemcpyAsync(out_host, os, ob, cudaMemcpyDeviceToHost, ctx->d2h) != cudaSuccess ||
      cudaEventRecord(ctx->ev_free[k], ctx->d2h) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  ctx->slot = (k + 1) % kHostSlots;
  return COLIBRI_OK;
}

int colibri_moe_host_sync(colibri_moe_t* ctx) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  if (cudaStreamSynchronize(ctx->h2d) != cudaSuccess || cudaStreamSynchronize(ctx->d2h) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  return COLIBRI_OK;
}

// ------------------------------------------------------------------------- expert parallelism

int colibri_moe_ep_dispatch(colibri_moe_t* ctx, const void* x, int32_t T, void* send_rows, int32_t* send_counts,
                            void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size == 0) return COLIBRI_ERR_UNSUPPORTED;
  if (T < 0 || T > ctx->cfg.max_tokens) return COLIBRI_ERR_INVALID_ARG;
  if (!ctx->loaded) return COLIBRI_ERR_STATE;
  if (!send_counts || !is_device_ptr(send_counts, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  const colibri_moe_config_t& c = ctx->cfg;
  const int E = c.num_experts, d = c.d_model, k = ctx->k;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (cudaMemsetAsync(send_counts, 0, E * sizeof(int32_t), s) != cudaSuccess) {
      cudaGetLastError();
      return COLIBRI_ERR_CUDA;
    }
    ctx->last_T = 0;
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!x || !send_rows) return COLIBRI_ERR_INVALID_ARG;
  const size_t xb = static_cast<size_t>(T) * d * ctx->esize;
  const size_t sb = static_cast<size_t>(T) * k * d * ctx->esize;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(send_rows)) & 15) return COLIBRI_ERR_INVALID_ARG;
  if (overlap(x, xb, send_rows, sb) || overlap(send_counts, E * sizeof(int32_t), send_rows, sb))
    return COLIBRI_ERR_INVALID_ARG;
  if (!is_device_ptr(x, ctx->device) || !is_device_ptr(send_rows, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  const int nchunks = (T + kRouterChunk - 1) / kRouterChunk;
  RouterArgs ra{x, ctx->w_router, ctx->b_router, T, d, E, ctx->dchunk, ctx->idx, ctx->gate, ctx->row_of, ctx->hist,
                ctx->sched, k, c.gate_mode, 0, k, E, nullptr, ctx->tile_done, d / 128, ctx->split_part};
  const int rc = enqueue_router(ctx, ra, x, T, nchunks, s);
  if (rc) return rc;
  EpPackArgs pa{x, ctx->idx, ctx->row_of, ctx->hist, ctx->sched, T, d, E, k, send_rows, send_counts,
                &ctx->sched->status};
  if (launch_ep_pack(c.dtype, pa, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  ctx->last_T = T;
  ctx->last_kernels = 2;
  return COLIBRI_OK;
}

int colibri_moe_ep_experts(colibri_moe_t* ctx, const void* recv_rows, const int32_t* recv_counts, void* y_rows,
                           void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size == 0) return COLIBRI_ERR_UNSUPPORTED;
  if (!ctx->loaded) return COLIBRI_ERR_STATE;
  if (!recv_counts) return COLIBRI_ERR_INVALID_ARG;
  const colibri_moe_config_t& c = ctx->cfg;
  const int El = ctx->n_arena, N = ctx->ep_size, d = c.d_model, f = c.d_ff;
  // the plan: received rows are source-major (p, j); Xp segments expert-major (j, p), padded to 128
  EpPlan plan{};
  plan.n_seg = N * El;
  plan.El = El;
  int64_t R = 0;
  for (int p = 0; p < N; ++p)
    for (int j = 0; j < El; ++j) {
      const int32_t n = recv_counts[p * El + j];
      if (n < 0) return COLIBRI_ERR_INVALID_ARG;
      plan.src[p * El + j] = static_cast<int32_t>(R < INT32_MAX ? R : INT32_MAX);
      plan.counts[j] += n;
      R += n;
    }
  if (R > ctx->ep_max_rows) return COLIBRI_ERR_INVALID_ARG;
  {
    int32_t off = 0, mt = 0;
    for (int j = 0; j < El; ++j) {
      plan.offsets[j] = off;
      plan.mstart[j] = mt;
      int32_t fill = off;
      for (int p = 0; p < N; ++p) {
        plan.dst[p * El + j] = fill;
        fill += recv_counts[p * El + j];
      }
      const int32_t tiles = (plan.counts[j] + kRowTile - 1) / kRowTile;
      off += tiles * kRowTile;
      mt += tiles;
    }
    plan.offsets[El] = off;
    plan.mstart[El] = mt;
  }
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  if (R == 0) {
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!recv_rows || !y_rows) return COLIBRI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(recv_rows) | reinterpret_cast<uintptr_t>(y_rows)) & 15)
    return COLIBRI_ERR_INVALID_ARG;
  if (overlap(recv_rows, static_cast<size_t>(R) * d * ctx->esize, y_rows, static_cast<size_t>(R) * d * 4))
    return COLIBRI_ERR_INVALID_ARG;
  if (!is_device_ptr(recv_rows, ctx->device) || !is_device_ptr(y_rows, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = c.dtype == COLIBRI_DTYPE_BF16;
  const bool swiglu = c.act == COLIBRI_ACT_SWIGLU;
  // CTA-pair GEMMs: the down projection writes each row straight into y_rows at its receive index
  // (tok_of_row holds it; an expert rank has no other use for it); other kernels write Y and an
  // unregroup kernel copies it back
  const bool direct_y = bf16 && ctx->pair_gemm;
  EpRegroupArgs rg{recv_rows, ctx->xp, static_cast<int>(R), static_cast<int>(d * ctx->esize), ctx->ep_sched, plan,
                   direct_y ? ctx->tok_of_row : nullptr};
  if (launch_ep_regroup(rg, ctx->num_sms, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  int64_t max_mtiles = (R + (kRowTile - 1) * static_cast<int64_t>(El)) / kRowTile;
  if (max_mtiles > ctx->rows_alloc / kRowTile) max_mtiles = ctx->rows_alloc / kRowTile;
  Sched* const sc = ctx->ep_sched;
  int32_t* const status = &ctx->sched->status;
  // the weight-major GEMMs for few rows per local expert (the received counts are known here)
  const int wm_nt = bf16 && ctx->pair_gemm ? wm_tile_rows_for(ctx, R / El, R, El) : 0;
  const bool wm_one = wm_nt > 0 && ctx->wm_fused && ctx->dynamic_tiles;
  if (wm_nt > 0) {
    const int64_t tok_tiles = R / wm_nt + El;
    WmMaps mu, md;
    mu.w = swiglu ? ctx->tm_w13_half : ctx->tm_w13_dec;
    md.w = ctx->tm_w2_dec;
    for (int i = 0; i < kWmTokMaps; ++i) {
      mu.tok[i] = ctx->tm_xp_dec[i];
      md.tok[i] = ctx->tm_h_dec[i];
    }
    GemmArgs up{sc, El, d, ctx->n_up, 0, ctx->h, f, ctx->b1, f, ctx->timeout_ns, status, nullptr, nullptr, nullptr,
                ctx->dynamic_tiles ? &sc->tile_ctr[0] : nullptr, nullptr, 0, nullptr, 0};
    up.wm_ntok = wm_nt;
    // the down projection writes each row at its receive index (tok_of_row, filled by the regroup)
    GemmArgs dn{sc, El, f, d, 0, y_rows, d, ctx->b2, d, ctx->timeout_ns, status, nullptr, nullptr, nullptr,
                ctx->dynamic_tiles ? &sc->tile_ctr[1] : nullptr, nullptr, 0, nullptr, 0, ctx->tok_of_row};
    dn.wm_ntok = wm_nt;
    const int64_t ctas_up = 2 * (ctx->n_up / 256) * tok_tiles, ctas_dn = 2 * (d / 256) * tok_tiles;
    const int epi_up = swiglu ? kEpiSwiGLU : kEpiReluBias;
    if (wm_one) {
      WmFused fz;
      fz.maps[0] = mu;
      fz.maps[1] = md;
      fz.args[0] = up;
      fz.args[1] = dn;
      const int64_t ctas = ctas_up + ctas_dn;
      if (launch_wm_fused(epi_up, kEpiStoreF32, fz, static_cast<int>(ctas < ctx->wm_ctas ? ctas : ctx->wm_ctas), s) !=
          cudaSuccess)
        return COLIBRI_ERR_CUDA;
    } else {
      if (launch_wm_gemm(epi_up, mu, up, static_cast<int>(ctas_up < ctx->wm_ctas ? ctas_up : ctx->wm_ctas), s) !=
              cudaSuccess ||
          launch_wm_gemm(kEpiStoreF32, md, dn, static_cast<int>(ctas_dn < ctx->wm_ctas ? ctas_dn : ctx->wm_ctas), s) !=
              cudaSuccess)
        return COLIBRI_ERR_CUDA;
    }
  } else if (bf16 && ctx->pair_gemm) {
    const int bn = tc_gemm_block_n();
    const int64_t max_pairs = (max_mtiles + El + 1) / 2;
    GemmArgs up{sc, El, d, ctx->n_up, ctx->n_up / bn, ctx->h, f, ctx->b1, f, ctx->timeout_ns, status, nullptr, nullptr,
                nullptr, ctx->dynamic_tiles ? &sc->tile_ctr[0] : nullptr, nullptr, 0, nullptr, ctx->half_tiles ? 1 : 0};
    int64_t ctas = 2 * max_pairs * up.n_tiles;
    int grid = static_cast<int>(ctas < ctx->pair_ctas ? ctas : ctx->pair_ctas);
    if (launch_pair_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, false, ctx->tm_xp, ctx->tm_xp_dec[kBox64], ctx->tm_w13_dec, up,
                         grid, s) !=
        cudaSuccess)
      return COLIBRI_ERR_CUDA;
    GemmArgs dn{sc, El, f, d, d / bn, y_rows, d, ctx->b2, d, ctx->timeout_ns, status, nullptr, nullptr, nullptr,
                ctx->dynamic_tiles ? &sc->tile_ctr[1] : nullptr, nullptr, 0, nullptr, ctx->half_tiles ? 1 : 0,
                ctx->tok_of_row};
    ctas = 2 * max_pairs * dn.n_tiles;
    grid = static_cast<int>(ctas < ctx->pair_ctas ? ctas : ctx->pair_ctas);
    if (launch_pair_gemm(kEpiStoreF32, false, ctx->tm_h, ctx->tm_h_dec[kBox64], ctx->tm_w2_dec, dn, grid, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
  } else if (bf16) {
    const int bn = tc_gemm_block_n();
    GemmArgs up{sc, El, d, ctx->n_up, ctx->n_up / bn, ctx->h, f, ctx->b1, f, ctx->timeout_ns, status, nullptr, nullptr,
                nullptr, nullptr, nullptr, 0};
    int64_t tiles = max_mtiles * up.n_tiles;
    int grid = static_cast<int>(tiles < ctx->num_sms ? tiles : ctx->num_sms);
    if (launch_tc_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, false, ctx->tm_xp, ctx->tm_w13, up, grid, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    GemmArgs dn{sc, El, f, d, d / bn, ctx->y, d, ctx->b2, d, ctx->timeout_ns, status, nullptr, nullptr, nullptr,
                nullptr, nullptr, 0};
    tiles = max_mtiles * dn.n_tiles;
    grid = static_cast<int>(tiles < ctx->num_sms ? tiles : ctx->num_sms);
    if (launch_tc_gemm(kEpiStoreF32, false, ctx->tm_h, ctx->tm_w2, dn, grid, s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
  } else {
    SimtGemmArgs up{sc, El, d, f, static_cast<const float*>(ctx->xp), static_cast<const float*>(ctx->w13),
                    static_cast<const float*>(ctx->w3), ctx->b1, static_cast<float*>(ctx->h)};
    if (launch_simt_gemm(swiglu ? kEpiSwiGLU : kEpiReluBias, up, static_cast<int>(max_mtiles), s) != cudaSuccess)
      return COLIBRI_ERR_CUDA;
    SimtGemmArgs dn{sc, El, f, d, static_cast<const float*>(ctx->h), static_cast<const float*>(ctx->w2), nullptr,
                    ctx->b2, ctx->y};
    if (launch_simt_gemm(kEpiStoreF32, dn, static_cast<int>(max_mtiles), s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  }
  if (!direct_y) {
    EpUnregroupArgs ug{ctx->y, static_cast<float*>(y_rows), static_cast<int>(R), d, plan};
    if (launch_ep_unregroup(ug, ctx->num_sms, s) != cudaSuccess) return COLIBRI_ERR_CUDA;
  }
  ctx->last_kernels = (direct_y ? 3 : 4) - (wm_one ? 1 : 0);
  ctx->last_gemm = wm_one ? COLIBRI_GEMM_WEIGHT_MAJOR_FUSED
                   : wm_nt > 0 ? COLIBRI_GEMM_WEIGHT_MAJOR
                   : !bf16 ? COLIBRI_GEMM_SIMT
                   : ctx->pair_gemm ? COLIBRI_GEMM_PAIR : COLIBRI_GEMM_SINGLE_CTA;
  return COLIBRI_OK;
}

int colibri_moe_ep_combine(colibri_moe_t* ctx, const float* y_back, void* out, void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->ep_size == 0) return COLIBRI_ERR_UNSUPPORTED;
  if (ctx->last_T < 0) return COLIBRI_ERR_STATE;
  const int T = ctx->last_T, d = ctx->cfg.d_model;
  if (T == 0) {
    ctx->last_kernels = 0;
    ctx->last_gemm = COLIBRI_GEMM_NONE;
    return COLIBRI_OK;
  }
  if (!y_back || !out) return COLIBRI_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(y_back) | reinterpret_cast<uintptr_t>(out)) & 15) return COLIBRI_ERR_INVALID_ARG;
  if (overlap(y_back, static_cast<size_t>(T) * ctx->k * d * 4, out, static_cast<size_t>(T) * d * ctx->out_esize))
    return COLIBRI_ERR_INVALID_ARG;
  if (!is_device_ptr(y_back, ctx->device) || !is_device_ptr(out, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  CombineArgs ca{y_back, ctx->row_of, ctx->gate, T, d, out, ctx->k};
  if (launch_combine(ctx->cfg.out_dtype, ca, ctx->num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return COLIBRI_ERR_CUDA;
  ctx->last_kernels = 1;
  return COLIBRI_OK;
}

int colibri_moe_get_routing(colibri_moe_t* ctx, int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                            int32_t* row_of, void* stream) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (ctx->last_T < 0) return COLIBRI_ERR_STATE;
  const void* ptrs[5] = {idx, gate, counts, offsets, row_of};
  for (const void* p : ptrs)
    if (p && !is_device_ptr(p, ctx->device)) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t T = static_cast<size_t>(ctx->last_T), E = ctx->cfg.num_experts;
  const size_t k = ctx->k, S = ctx->S;
  bool ok = true;
  // the routed slots [T, k] of the internal [T, S] arrays (slot k is the shared expert)
  auto copy_slots = [&](void* dst, const void* src) {
    return cudaMemcpy2DAsync(dst, k * 4, src, S * 4, k * 4, T, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  };
  if (idx && T) ok = ok && copy_slots(idx, ctx->idx);
  if (gate && T) ok = ok && copy_slots(gate, ctx->gate);
  if (row_of && T) ok = ok && copy_slots(row_of, ctx->row_of);
  if (T == 0) {
    if (counts) ok = ok && cudaMemsetAsync(counts, 0, E * 4, s) == cudaSuccess;
    if (offsets) ok = ok && cudaMemsetAsync(offsets, 0, (E + 1) * 4, s) == cudaSuccess;
  } else {
    if (counts)
      ok = ok && cudaMemcpyAsync(counts, ctx->sched->counts, E * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
    if (offsets)
      ok = ok &&
           cudaMemcpyAsync(offsets, ctx->sched->offsets, (E + 1) * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  }
  if (!ok) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  return COLIBRI_OK;
}

int colibri_moe_debug_buffer(colibri_moe_t* ctx, int32_t which, void** ptr, int64_t* rows) {
  if (!ctx || !ptr) return COLIBRI_ERR_INVALID_ARG;
  void* p = nullptr;
  switch (which) {
    case 0: p = ctx->xp; break;
    case 1: p = ctx->h; break;
    case 2: p = ctx->y; break;
    case 3: p = ctx->tok_of_row; break;
    default: return COLIBRI_ERR_INVALID_ARG;
  }
  *ptr = p;
  if (rows) *rows = ctx->rows_alloc;
  return COLIBRI_OK;
}

int colibri_moe_num_stages(const colibri_moe_t* ctx, int32_t* n_stages) {
  if (!ctx || !n_stages) return COLIBRI_ERR_INVALID_ARG;
  *n_stages = kNumStages;
  return COLIBRI_OK;
}

int colibri_moe_last_kernel_count(const colibri_moe_t* ctx, int32_t* n) {
  if (!ctx || !n) return COLIBRI_ERR_INVALID_ARG;
  *n = ctx->last_kernels;
  return COLIBRI_OK;
}

int colibri_moe_last_gemm(const colibri_moe_t* ctx, int32_t* kind) {
  if (!ctx || !kind) return COLIBRI_ERR_INVALID_ARG;
  *kind = ctx->last_gemm;
  return COLIBRI_OK;
}

int colibri_moe_set_stage_events(colibri_moe_t* ctx, void* const* events, int32_t n) {
  if (!ctx) return COLIBRI_ERR_INVALID_ARG;
  if (!events || n == 0) {
    ctx->events.clear();
    return COLIBRI_OK;
  }
  if (n != kNumStages + 1) return COLIBRI_ERR_INVALID_ARG;
  ctx->events.assign(reinterpret_cast<cudaEvent_t const*>(events), reinterpret_cast<cudaEvent_t const*>(events) + n);
  return COLIBRI_OK;
}

int colibri_moe_probe_wait_timeout(colibri_moe_t* ctx, int32_t timeout_us, void* stream) {
  if (!ctx || timeout_us < 1 || timeout_us > 1000000) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  if (launch_wait_probe(&ctx->sched->status, static_cast<uint64_t>(timeout_us) * 1000ull,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  return COLIBRI_OK;
}

int colibri_moe_device_status(colibri_moe_t* ctx, int32_t* status) {
  if (!ctx || !status) return COLIBRI_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return COLIBRI_ERR_CUDA;
  int32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&v, &ctx->sched->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(&ctx->sched->status, 0, 4) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return COLIBRI_ERR_CUDA;
  }
  *status = v;
  return COLIBRI_OK;
}

}  // extern "C"
