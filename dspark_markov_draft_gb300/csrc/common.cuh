// Device helpers shared by the walk kernels: bf16 handling, Philox4x32-10 Gumbel
// noise, the orderable argmax word, the device status word, the workspace layout and
// the bounded grid-wide step exchange.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/dspark.h"

namespace dspark {

constexpr int kRank = DSPARK_RANK;
constexpr uint32_t kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------- bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---------------------------------------------------------------- Philox / Gumbel

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32->64
// multiplies whose halves are xored with the other two words and the round key; the
// key advances by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The four words for vocabulary entries 4m .. 4m+3 of draft position i, row b.
__device__ __forceinline__ uint4 philox_block(uint64_t seed, int b, int i, uint32_t m) {
  return philox4x32_10(make_uint4(m, static_cast<uint32_t>(i), static_cast<uint32_t>(b), 0u),
                       static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

__device__ __forceinline__ uint32_t uint4_get(const uint4& w, int j) {
  return j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
}

// -ln(u) for u in (0, 1) with a small RELATIVE error everywhere, including u -> 1
// where the largest Gumbel values come from:
//   * u <= 0.75: -log2(u) ln 2 from the hardware base-2 logarithm; |log2 u| >= 0.41
//     there, so its ~2^-22 error is below 6e-7 relative;
//   * u > 0.75: t = 1 - u is exact, and -ln(1 - t) = 2 atanh(s) with s = t / (2 - t)
//     in (0, 1/7], summed as the series 2 s (1 + s^2/3 + s^4/5 + s^6/7) (the first
//     omitted term is below 3e-15 relative).
__device__ __forceinline__ float neg_log_unit(float u) {
  float l2, r;
  asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(u));
  const float a = -l2 * 0.693147180559945f;
  const float t = 1.f - u;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(2.f - t));
  const float sv = t * r;
  const float s2 = sv * sv;
  const float poly = fmaf(s2, fmaf(s2, fmaf(s2, 0.142857142857143f, 0.2f), 0.333333333333333f), 1.f);
  const float b = 2.f * sv * poly;
  return u > 0.75f ? b : a;
}

// u = (2 * (w >> 9) + 1) * 2^-24 lies strictly inside (0, 1) and is exact in fp32;
// g = -ln(-ln(u)): the inner logarithm as above, the outer one (argument in
// [6e-8, 16.7]) from the hardware base-2 logarithm, absolute error below 5e-6.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  // (1 + x 2^-23) - 1 is exact (both in [1, 2)) and adding 2^-24 to x 2^-23 is exact for
  // x < 2^23, so this is the same u without an integer-to-float conversion.
  const float f = __uint_as_float(0x3F800000u | (w >> 9));
  const float u = __fadd_rn(__fsub_rn(f, 1.0f), 5.9604644775390625e-08f);
  float l2;
  asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(neg_log_unit(u)));
  return -l2 * 0.693147180559945f;
}

// ---------------------------------------------------------------- argmax words

// Monotone map of fp32 to uint32 for the max reduction. NaN maps above every number
// (so a NaN wins) and -0 maps to the key of +0 (so they tie).
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;  // NaN
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;                         // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One 64-bit word per candidate: key in the high half, the complement of the index
// in the low half, so the integer maximum is the largest key and, among equal keys,
// the smallest index (torch.argmax order).
__device__ __forceinline__ uint64_t pack_best(uint32_t key, uint32_t idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ int32_t unpack_idx(uint64_t word) {
  return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(word));
}
__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint64_t warp_max64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = umax64(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// ---------------------------------------------------------------- status and memory

__device__ __forceinline__ void report(int32_t* status_dev, int32_t code) {
  if (status_dev) atomicCAS(status_dev, 0, code);
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- workspace

// Workspace layout (bytes), shared by the dense and the top-k walk:
//   [0, 256)                 header: abort flag, exit counter
//   [256, 256 + 128*K)       per-step arrival counters, one 128-byte line each
//   next 8*K*bs              per-step argmax words slot[i][b]
//   next (aligned to 256)    top-k candidate lists int32 [bs, K, top_k]
//   next (aligned to 256)    their base logits fp32 [bs, K, top_k]
struct WsHeader {
  uint32_t abort;
  uint32_t exit_count;
};
constexpr size_t kWsHeader = 256;
constexpr size_t kWsCounterStride = 128;

__host__ __device__ inline size_t ws_counters_off() { return kWsHeader; }
__host__ __device__ inline size_t ws_slots_off(int K) {
  return kWsHeader + kWsCounterStride * static_cast<size_t>(K);
}
__host__ __device__ inline size_t ws_cand_off(int K, int bs) {
  const size_t end = ws_slots_off(K) + 8ull * K * bs;
  return (end + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ inline size_t ws_cand_base_off(int K, int bs, int top_k) {
  const size_t end = ws_cand_off(K, bs) + 4ull * bs * K * static_cast<size_t>(top_k);
  return (end + 255) & ~static_cast<size_t>(255);
}
__host__ __device__ inline size_t ws_total(int K, int bs, int top_k) {
  return ws_cand_base_off(K, bs, top_k) + 4ull * bs * K * static_cast<size_t>(top_k);
}

// Programmatic dependent launch: wait until the previous kernel in the stream has
// completed and its writes are visible (a no-op for a kernel launched in plain stream
// order).
__device__ __forceinline__ void wait_previous_kernel() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- step exchange

struct StepSync {
  WsHeader* hdr;
  uint32_t* counters;  // stride kWsCounterStride bytes
  uint64_t* slots;     // [K][bs]
  int32_t* status_dev;
  uint32_t grid;
  uint64_t timeout_ns;
  uint32_t flags;

  __device__ __forceinline__ uint32_t* counter(int i) const {
    return reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(counters) + kWsCounterStride * i);
  }
};

// Give up a wait: flag the abort for the other CTAs and report a timeout.
__device__ __forceinline__ void give_up(const StepSync& s) {
  atomicExch(&s.hdr->abort, 1u);
  report(s.status_dev, DSPARK_ERR_TIMEOUT);
}

// Exchange of the per-row argmax words of step i. best_s[b] (shared memory, b < bs)
// holds this CTA's word on entry and the grid-wide maximum on return.
// Each row's word goes into slot[i][b] with one 64-bit atomicMax; thread 0 then
// arrives at the step counter with a release add (ordering the CTA's atomics before
// it), spins with acquire loads until the whole grid has arrived, and the winners are
// read back. Every thread of the CTA calls it. The spin is bounded by timeout_ns of
// wall-clock time and watches the workspace abort flag; on either, the wait gives up
// and false is returned (the same value in every thread), and the caller returns from
// the kernel.
// The exchange in two halves, for kernels with work to do while the grid arrives:
// exchange_arrive publishes this CTA's words and arrives at the step counter;
// exchange_wait waits for the grid and reads the winners back.
__device__ __forceinline__ void exchange_arrive(const StepSync& s, int i, int bs, bool skip_arrival,
                                                const uint64_t* best_s) {
  __syncthreads();
  if (threadIdx.x < bs && best_s[threadIdx.x] != 0ull)
    atomicMax(reinterpret_cast<unsigned long long*>(s.slots + static_cast<size_t>(i) * bs + threadIdx.x),
              static_cast<unsigned long long>(best_s[threadIdx.x]));
  __syncthreads();
  if (threadIdx.x == 0 && !skip_arrival)
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(s.counter(i)) : "memory");
}
__device__ __forceinline__ bool exchange_wait(const StepSync& s, int i, int bs, uint64_t* best_s,
                                              int* sh_flag) {
  if (threadIdx.x == 0) {
    bool failed = false;
    uint32_t* ctr = s.counter(i);
    uint64_t t0 = 0;
    uint32_t it = 0;
    while (ld_acquire_u32(ctr) < s.grid) {
      if ((++it & 63u) != 0u) continue;
      if (t0 == 0) t0 = globaltimer_ns();
      if (*reinterpret_cast<volatile uint32_t*>(&s.hdr->abort) != 0u) { failed = true; break; }
      if (globaltimer_ns() - t0 > s.timeout_ns) { give_up(s); failed = true; break; }
    }
    *sh_flag = failed ? 0 : 1;
  }
  __syncthreads();
  if (*sh_flag == 0) return false;
  if (threadIdx.x < bs) best_s[threadIdx.x] = ld_relaxed_u64(s.slots + static_cast<size_t>(i) * bs + threadIdx.x);
  __syncthreads();
  return true;
}

__device__ __forceinline__ bool exchange_best(const StepSync& s, int i, int bs,
                                              bool skip_arrival, uint64_t* best_s,
                                              int* sh_flag) {
  __syncthreads();
  if (threadIdx.x < bs && best_s[threadIdx.x] != 0ull)
    atomicMax(reinterpret_cast<unsigned long long*>(s.slots + static_cast<size_t>(i) * bs + threadIdx.x),
              static_cast<unsigned long long>(best_s[threadIdx.x]));
  __syncthreads();
  if (threadIdx.x == 0) {
    bool failed = false;
    uint32_t* ctr = s.counter(i);
    // the release add is cumulative: the CTA barrier above orders every thread's
    // atomicMax before it, so no separate fence is needed
    if (!skip_arrival) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
    uint64_t t0 = 0;
    uint32_t it = 0;
    while (ld_acquire_u32(ctr) < s.grid) {
      if ((++it & 63u) != 0u) continue;
      if (t0 == 0) t0 = globaltimer_ns();
      if (*reinterpret_cast<volatile uint32_t*>(&s.hdr->abort) != 0u) { failed = true; break; }
      if (globaltimer_ns() - t0 > s.timeout_ns) { give_up(s); failed = true; break; }
    }
    *sh_flag = failed ? 0 : 1;
  }
  __syncthreads();
  if (*sh_flag == 0) return false;
  if (threadIdx.x < bs) best_s[threadIdx.x] = ld_relaxed_u64(s.slots + static_cast<size_t>(i) * bs + threadIdx.x);
  __syncthreads();
  return true;
}

// Reset-behind: once every CTA has passed step i's barrier nobody reads step i-1's
// counter or slots again, so CTA 0 zeroes them for the next call.
__device__ __forceinline__ void reset_behind(const StepSync& s, int i, int bs) {
  if (blockIdx.x != 0 || i < 1) return;
  for (int t = threadIdx.x; t < bs; t += blockDim.x) s.slots[static_cast<size_t>(i - 1) * bs + t] = 0ull;
  if (threadIdx.x == 0) *s.counter(i - 1) = 0u;
}

// The last CTA to finish zeroes the final step's counter and slots and the exit counter.
__device__ __forceinline__ void finish_walk(const StepSync& s, int K, int bs, int* sh_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    *sh_flag = (atomicAdd(&s.hdr->exit_count, 1u) == s.grid - 1) ? 1 : 0;
  }
  __syncthreads();
  if (*sh_flag) {
    __threadfence();
    for (int t = threadIdx.x; t < bs; t += blockDim.x) s.slots[static_cast<size_t>(K - 1) * bs + t] = 0ull;
    if (threadIdx.x == 0) {
      *s.counter(K - 1) = 0u;
      s.hdr->exit_count = 0u;
    }
  }
}

}  // namespace dspark
