// Gathered A operand for the up-projection GEMMs: each 128-row A tile is filled straight from the
// token rows x[T, K] through token_of_row, so the expert-contiguous copy Xp is never written
// (hnwysp.cn/news/30485 2.2: hand the expert the token's row instead of copying it).
//
// kGatherWarps "gather" warps per CTA copy the tile with 16-byte cp.async (L2 only): lane l of
// gather warp w owns the 16-byte chunk (l % 8) of rows 4w + l/8 + kRowStep*i, so each warp
// instruction moves four whole 128-byte row pieces.  Chunks land where a 128-byte-swizzled TMA
// box would put them (chunk c of row r at c ^ (r % 8)), which is the layout the tcgen05
// shared-memory descriptors describe; since r % 8 is the same for all of a thread's rows, its
// destination offsets differ by whole 1024-byte swizzle atoms.
//
// Completion: every gather thread ends a stage with cp.async.mbarrier.arrive.noinc on a local
// `gfull` barrier (kGatherThreads expected arrivals), so the hardware signals the stage as soon
// as its rows land, with no thread blocking on it.  A forwarder thread waits on gfull, issues
// fence.proxy.async (the rows were written through the generic proxy, the tensor cores read them
// through the async proxy) and arrives on the MMA's `full` barrier.
//
// Measured on GB300 at the Mixtral-8x7B prefill shape, this path keeps the tensor pipe busy 77 %
// of the time against 91 % for the TMA-fed GEMM over Xp (the up GEMM 5-7 % slower, more than the
// 30 us the skipped copy saves), so it is built but not the default.  Neither a seventh stage,
// a second forwarder nor four gather warps changed that; an earlier form with TMA tile::gather4
// (one instruction per 4 rows) ran at about a third of the speed.
#pragma once
#include "tcgen05_ptx.cuh"

namespace colibri {
using ptx::cp_async_16;

constexpr int kGatherWarps = 2;
constexpr int kGatherThreads = 32 * kGatherWarps;
constexpr int kForwarders = 1;  // forwarder warps; divides the stage count of both GEMM kernels
constexpr int kGatherWarp0 = 6;                            // after producer, MMA and 4 epilogue warps
constexpr int kForwardWarp0 = kGatherWarp0 + kGatherWarps;
constexpr int kRowStep = 4 * kGatherWarps;             // rows between a thread's consecutive rows
constexpr int kGatherRows = 128 / kRowStep;            // rows per thread per tile
static_assert(kRowStep % 8 == 0, "a thread's rows share one position inside the 8-row swizzle atom");

struct AGather {
  const char* x;       // token rows, bf16 [T, K]
  size_t row_bytes;    // K * 2
  uint32_t dst_off;    // first row of this thread inside the tile, swizzled chunk
  int chunk_bytes;     // (lane % 8) * 16: the chunk's offset inside the 128-byte row piece
  int row0;            // 4w + lane / 8
  int tok[kGatherRows];       // tokens of the current tile's rows
  int tok_next[kGatherRows];  // tokens of the next tile's rows, loaded one tile ahead

  __device__ __forceinline__ void init(const void* x_, int K, int gw, int lane) {
    x = static_cast<const char*>(x_);
    row_bytes = static_cast<size_t>(K) * 2;
    row0 = 4 * gw + (lane >> 3);
    const int chunk = lane & 7;
    chunk_bytes = chunk * 16;
    dst_off = static_cast<uint32_t>(row0 * 128 + ((chunk ^ (row0 & 7)) * 16));
  }
  // Rows a_row .. a_row + 127 of the expert-ordered layout; rows at or past seg_end (padding, or the
  // second tile of a pair past the expert's rows) read token 0: computed, never stored.
  // Loads into tok_next; the loads are consumed one tile later, so their latency is hidden.
  __device__ __forceinline__ void prefetch_tokens(const int32_t* token_of_row, int a_row, int seg_end) {
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i) {
      const int r = a_row + row0 + kRowStep * i;
      tok_next[i] = r < seg_end ? token_of_row[r] : 0;
    }
  }
  __device__ __forceinline__ void advance_tile() {
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i) tok[i] = tok_next[i];
  }
  // The 64-wide K block kb of every row into the tile at shared address sA (1024-byte aligned).
  __device__ __forceinline__ void issue(uint32_t sA, int kb) const {
    const char* src = x + static_cast<size_t>(kb) * 128 + chunk_bytes;
#pragma unroll
    for (int i = 0; i < kGatherRows; ++i)
      cp_async_16(sA + dst_off + static_cast<uint32_t>(i * kRowStep * 128), src + static_cast<size_t>(tok[i]) * row_bytes);
  }
};

}  // namespace colibri
