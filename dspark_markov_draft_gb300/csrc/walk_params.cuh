// Kernel parameter blocks and launch plans of the walk kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace dspark {

struct WalkParams {
  const uint16_t* base;      // [bs, K, V] bf16
  const uint16_t* w1;        // [V, 256] bf16
  const uint16_t* w2;        // [V, 256] bf16 (bf16 path)
  const int8_t* w2q;         // [V, 256] int8 (int8 path)
  const float* scales;       // [V]
  const int32_t* prev;       // [bs]
  const uint64_t* seeds;     // [bs]
  int32_t* tokens;           // [bs, K]
  uint16_t* logits;          // [bs, K, V] bf16 or null
  const int32_t* cand;       // top-k candidates [bs, K, top_k] (top-k walk)
  const float* cand_base;    // their base logits [bs, K, top_k] fp32, or null (read from base)
  int64_t V;
  int32_t bs, K, top_k;
  float temperature;
  int32_t temp_is_one;
  int32_t resident_rows;     // W2 rows per CTA kept in shared memory (multiple of 32)
  int32_t slice_cap;         // upper bound of the rows of one CTA's vocabulary slice
  int32_t w2_tma;            // w2_map is valid (tensor-core walk)
  int32_t base_tma;          // base_map is valid (tensor-core walk)
  float inv_temperature;     // 1 / temperature, rounded to fp32 (tensor-core walk)
  const float* temps;        // [bs] per-row temperatures, or null (then `temperature`)
  const int32_t* modes;      // [bs] per-row modes, or null (then the kernel's mode)
  StepSync sync;
  // Tensor map over the W2 rows (int8 [V][256] or bf16 [V][256]), box of 32 rows x 128
  // bytes with the 128-byte swizzle: the tensor-core walk copies its shared-memory
  // resident rows with it, 32 rows and one 128-byte part of the row per copy.
  CUtensorMap w2_map;        // 128-byte aligned type
  // Tensor map over the base logits [bs][K][V] (bf16), box of 128 vocabulary rows x 1
  // position x N requests: one copy stages a tile's base logits for every request.
  CUtensorMap base_map;
};

// Per-row sampling settings. A PROB kernel serves batches with at least one sampled
// row: row b is sampled unless the per-row modes say greedy.
__device__ __forceinline__ bool row_sampled(const WalkParams& p, bool prob_kernel, int b) {
  return prob_kernel && (!p.modes || p.modes[b] == DSPARK_PROBABILISTIC);
}
__device__ __forceinline__ float row_temperature(const WalkParams& p, int b) {
  return p.temps ? p.temps[b] : p.temperature;
}
// Valid settings of row b: a known mode, and T > 0 and finite if the row is sampled.
__device__ __forceinline__ bool row_settings_ok(const WalkParams& p, bool prob_kernel, int b) {
  if (p.modes && p.modes[b] != DSPARK_GREEDY && p.modes[b] != DSPARK_PROBABILISTIC) return false;
  if (!row_sampled(p, prob_kernel, b)) return true;
  const float T = row_temperature(p, b);
  return T > 0.f && T < 3.4e38f;
}

// Threads per CTA of the persistent walk kernels: 16 warps.
constexpr int kWalkThreads = 512;
constexpr int kWalkWarps = kWalkThreads / 32;

// Shared memory outside the resident W2 rows, per CTA.
__host__ __device__ inline size_t walk_cc_fixed_smem(int bs, bool int8, int slice_cap) {
  return (int8 ? static_cast<size_t>(slice_cap) * 4 : 0)  // scales of the slice
         + static_cast<size_t>(bs) * kRank * 2            // W1[prev] rows, bf16
         + (int8 ? static_cast<size_t>(bs) * 3 * 64 * 4 : 0)  // their limb words
         + 64 * 4                                         // e-shift per row (int8 path)
         + 64 * 4                                         // prev tokens
         + 64 * 8                                         // per-row argmax words
         + kWalkWarps * 8 + 64                            // reduction scratch, flags
         + 256;                                           // alignment slack
}

// Prefetch this CTA's base-logit slices of position i (all rows) towards L2.
__device__ __forceinline__ void prefetch_base_slice(const WalkParams& p, int64_t v0, int n, int i) {
  if (i >= p.K || n <= 0) return;
  const int lines = (n * 2 + 127) / 128 + 1;
  for (int t = threadIdx.x; t < lines * p.bs; t += blockDim.x) {
    const int b = t / lines, l = t % lines;
    const uint16_t* row = p.base + (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v0;
    const int64_t off = min(static_cast<int64_t>(l) * 64, static_cast<int64_t>(n - 1));
    prefetch_l2(row + off);
  }
}

// Vocabulary slice of CTA c: starts are multiples of 32 (so a group of 4 consecutive
// entries never straddles two CTAs), the last slice ends at V.
__host__ __device__ inline int64_t slice_start(int c, int G, int64_t V) {
  if (c <= 0) return 0;
  if (c >= G) return V;
  return (static_cast<int64_t>(c) * V / G) & ~static_cast<int64_t>(31);
}

// Tensor-core walk: six warpgroups -- 4 producer warps, 16 epilogue warps, and a last
// warpgroup whose first warp issues the MMAs. The kernel is compiled for kTcLaunchRegs
// registers per thread (the most that 6 warps per SM sub-partition allow); the
// warpgroups then rebalance them with setmaxnreg: producers kTcProducerRegs, epilogue
// kTcEpilogueRegs, the issuing warpgroup kTcIssuerRegs. The shares add up to exactly
// the launch's total, so no request waits for registers that are not there.
constexpr int kTcProducerWarps = 4;
constexpr int kTcEpilogueWarps = 16;
constexpr int kTcThreads = (kTcProducerWarps + kTcEpilogueWarps + 4) * 32;
constexpr int kTcLaunchRegs = 80;
constexpr int kTcProducerRegs = 80;
constexpr int kTcEpilogueRegs = 88;
constexpr int kTcIssuerRegs = 48;
static_assert(kTcProducerWarps * 32 * kTcProducerRegs + kTcEpilogueWarps * 32 * kTcEpilogueRegs +
                      4 * 32 * kTcIssuerRegs ==
                  kTcThreads * kTcLaunchRegs,
              "the warpgroups' register shares must add up to the launch's registers");
// The epilogue keeps tile numbers in 8-bit fields, so a CTA's vocabulary slice holds at
// most kTcMaxTiles tiles of 128 rows.
constexpr int kTcMaxTiles = 255;

// Tensor-core walk: stages of base logits staged by tensor-map copies (128 rows x N
// requests, bf16, each).
__host__ __device__ constexpr int tc_base_stages(int N) { return N >= 64 ? 3 : 4; }
__host__ __device__ constexpr size_t tc_stage_ring_bytes(int N) {
  return static_cast<size_t>(tc_base_stages(N)) * 128 * N * 2;
}

// Tensor-core walk: shared memory besides the B operand, the base-logit stages, the
// slice's scales and the resident rows.
__host__ __device__ inline size_t walk_tc_misc_smem() {
  return 64 * 4          // prev tokens
         + 64 * 8        // seeds
         + 64 * 8        // per-row argmax words
         + 4 * 64 * 8    // per-quadrant argmax words
         + 2 * 8         // 2^-s as two factors
         + 64 * 4 + 8    // 1/T per row, greedy-row mask
         + 24 * 8 + 32;  // mbarriers, TMEM base, flags, batch |e| maximum
}

}  // namespace dspark
