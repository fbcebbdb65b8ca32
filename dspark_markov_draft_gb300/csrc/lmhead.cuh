// Parameters of the fused LM-head GEMM and top-k selection (lmhead.cu).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace dspark {

// Every kLmSampleStride-th LM-head row is scored in the sample pass.
constexpr int kLmSampleStride = 9;
// Flag: every row takes the exact path (testing).
constexpr int32_t kLmForceExact = 1;

struct LmParams {
  const uint16_t* hidden;    // [M, d] bf16
  const uint16_t* lm_head;   // [V, d] bf16
  int64_t V;
  int32_t M, d, k;
  int32_t S;                 // sampled LM-head rows
  int32_t cap;               // list capacity per hidden row
  float* sample;             // [M, S] sampled logits
  uint32_t* pivot;           // [M] pivot keys
  uint32_t* cnt;             // [M] list lengths
  uint64_t* list;            // [M, cap] packed {key, 2^32-1-v}
  int32_t* cand;             // out [M, k] candidate vocabulary ids
  float* cand_base;          // out [M, k] their logits
  int32_t* stats;            // optional [2]: rows on the exact path, rows whose list overflowed
  int32_t* status_dev;
  int32_t flags;
  uint64_t timeout_ns;
  CUtensorMap w_map;         // LM head [V][d], box 64 x 128 rows, 128-byte swizzle
  CUtensorMap ws_map;        // every kLmSampleStride-th LM-head row, same box
  CUtensorMap h_map;         // hidden [M][d], box 64 x 256 rows, 128-byte swizzle
};

// Workspace layout of the fused path (bytes, 256-aligned parts).
__host__ __device__ inline int32_t lm_samples(int64_t V) {
  return static_cast<int32_t>((V + kLmSampleStride - 1) / kLmSampleStride);
}
__host__ __device__ inline int32_t lm_cap(int32_t k) { return 3 * k + 1024; }
__host__ __device__ inline size_t lm_align(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
__host__ __device__ inline size_t lm_ws_sample(int32_t M, int64_t V) { return lm_align(4ull * M * lm_samples(V)); }
__host__ __device__ inline size_t lm_ws_total(int32_t M, int64_t V, int32_t k) {
  return lm_ws_sample(M, V) + 2 * lm_align(4ull * M) + lm_align(8ull * M * lm_cap(k));
}

}  // namespace dspark
