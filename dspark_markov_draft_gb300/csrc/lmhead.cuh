// Parameters of the fused LM-head GEMM and top-k selection (lmhead.cu).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace dspark {

// Every kLmSampleStride-th LM-head row is scored in the sample pass.
constexpr int kLmSampleStride = 16;
// Flag: every row takes the exact path (testing).
constexpr int32_t kLmForceExact = 1;

// The GEMM's CTA: warp 0 issues the tensor-map copies, warp 1 the MMAs, kLmEpiWarps
// warps read the accumulator (four per tensor-memory lane quadrant).
constexpr int kLmEpiWarps = 16;
constexpr int kLmThreads = (2 + kLmEpiWarps) * 32;
constexpr int kLmAStageBytes = 128 * 128;   // 128 LM-head rows x 64 bf16 of d
constexpr int kLmMaxStages = 6;

constexpr int kLmSmemLimit = 232448;        // opt-in dynamic shared memory per block
// After the stages: barriers (128 bytes) and each epilogue warp's column thresholds
// (4 steps x 32 floats).
constexpr int kLmTailBytes = 128 + kLmEpiWarps * 4 * 32 * 4;

// Hidden rows of a chunk (a multiple of 32, at most 512): part 0 = rows [0, n0) with
// n0 = min(256, rows), part 1 = rows [256, 256 + n1). The two CTAs of a pair each stage
// half of each part (lm_box0 and lm_box1 rows), as the paired MMA splits B along N.
__host__ __device__ inline int lm_b_rows(int32_t M) {
  const int m = M < 512 ? M : 512;
  return (m + 31) & ~31;
}
__host__ __device__ inline int lm_box0(int32_t M) { return (lm_b_rows(M) < 256 ? lm_b_rows(M) : 256) / 2; }
__host__ __device__ inline int lm_box1(int32_t M) { return (lm_b_rows(M) > 256 ? lm_b_rows(M) - 256 : 0) / 2; }
__host__ __device__ inline int lm_stage_bytes(int32_t M) { return kLmAStageBytes + 64 * lm_b_rows(M); }
__host__ __device__ inline int lm_stages(int32_t M) {
  const int n = (kLmSmemLimit - 1024 - kLmTailBytes) / lm_stage_bytes(M);
  return n < kLmMaxStages ? n : kLmMaxStages;
}
__host__ __device__ inline int lm_gemm_smem(int32_t M) {
  return 1024 + lm_stages(M) * lm_stage_bytes(M) + kLmTailBytes;
}

struct LmParams {
  const uint16_t* hidden;    // [M, d] bf16
  const uint16_t* lm_head;   // [V, d] bf16
  int64_t V;
  int32_t M, d, k;
  int32_t S;                 // sampled LM-head rows
  int32_t cap;               // list capacity per hidden row
  float* sample;             // [M, S] sampled logits
  uint32_t* pivot;           // [M] pivot keys
  uint32_t* cnt;             // [M] list lengths, at cnt[m * kLmCntStride]
  uint64_t* list;            // [M, cap] packed {key, 2^32-1-v}
  int32_t* cand;             // out [M, k] candidate vocabulary ids
  float* cand_base;          // out [M, k] their logits
  int32_t* stats;            // optional [2]: rows on the exact path, rows whose list overflowed
  int32_t* status_dev;
  int32_t flags;
  int32_t ksplit;            // sample pass: parts of d per tile, summed by fp32 atomics (1: stored)
  uint64_t timeout_ns;
  CUtensorMap w_map;         // LM head [V][d], box 64 x 128 rows, 128-byte swizzle
  CUtensorMap ws_map;        // every kLmSampleStride-th LM-head row, same box
  CUtensorMap h_map0;        // hidden [M][d], box 64 x lm_box0(M) rows, 128-byte swizzle
  CUtensorMap h_map1;        // hidden [M][d], box 64 x lm_box1(M) rows (when M > 256)
};

// Workspace layout of the fused path (bytes, 256-aligned parts).
__host__ __device__ inline int32_t lm_samples(int64_t V) {
  return static_cast<int32_t>((V + kLmSampleStride - 1) / kLmSampleStride);
}
__host__ __device__ inline int32_t lm_cap(int32_t k) { return 3 * k + 1024; }
__host__ __device__ inline size_t lm_align(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
__host__ __device__ inline size_t lm_ws_sample(int32_t M, int64_t V) { return lm_align(4ull * M * lm_samples(V)); }
// List counters: one per hidden row, each on its own 128-byte line (the filter pass's
// appends to different rows do not queue behind one another in L2).
constexpr int kLmCntStride = 32;
__host__ __device__ inline size_t lm_ws_cnt(int32_t M) { return lm_align(4ull * kLmCntStride * M); }
__host__ __device__ inline size_t lm_ws_total(int32_t M, int64_t V, int32_t k) {
  return lm_ws_sample(M, V) + lm_align(4ull * M) + lm_ws_cnt(M) + lm_align(8ull * M * lm_cap(k));
}

}  // namespace dspark
