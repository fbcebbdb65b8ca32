// Full-vocabulary Markov draft walk with the bias contraction on the 5th-generation
// tensor cores (tcgen05), for batches where W2 . E[256 x bs] is a real dense GEMM.
// Same method and per-position exchange as the CUDA-core walk (vLLM PR #62958,
// "Overview": one cooperative kernel for the whole walk, W2 on chip where it fits,
// one packed atomic per step for the cross-CTA argmax).
//
// Per CTA (one per SM, 16 warps) and per draft position:
//   * B operand: the bs embedding rows W1[prev_b] (N = 16, 32 or 64 rows, zero
//     padded), 16-bit, K-major, 128-byte swizzled in shared memory. With int8 W2 each
//     row is scaled by a power of two 2^s_b so that max|e| lies in [2^14, 2^15) and
//     converted to fp16 (exact for every bf16 value within 2^-28 of the row maximum;
//     inf and NaN stay inf and NaN); with bf16 W2 the rows are used as they are.
//   * A operand: 128 W2 rows per tile, written into tensor memory (tcgen05.st) by 8
//     producer warps: int8 codes become exact fp16 integers through a byte permute
//     with 0x64 exponent bytes and one packed subtract; bf16 rows are copied. Rows of
//     the slice that fit stay resident in shared memory (XOR-swizzled 16-byte chunks,
//     conflict-free for this access), brought in at position 0 with cp.async; the
//     rest are re-read from L2.
//   * D[128 x N] = A . B^T accumulates in fp32 in tensor memory. One thread issues an
//     MMA only about every 50 cycles whatever N is (up to 128), so the K range is
//     split in two halves issued by two threads: for N <= 32 into two accumulators
//     (issued concurrently, added by the epilogue), for N = 64 into one (half 1 issued
//     after half 0, ordered through an mbarrier and tensor-core fences).
//   * Epilogue (8 warps): thread = tensor-memory lane = one vocabulary row of the
//     tile, for N/2 request rows. It reads D (adding the K-half accumulators), forms
//     l = base + scale_v 2^-s D (base logits staged one tile ahead by a tensor-map
//     copy), the score (greedy: l; probabilistic: bf16(l)/T plus Gumbel noise, whose
//     Philox blocks of 4 consecutive rows are drawn once per lane quad and exchanged
//     by a 4 x 4 transpose), and keeps per column the running maximum and the tile
//     where it was first reached; lanes and quadrants are combined once per position.
//   * Producers, MMA issuers and the epilogue hand tiles over through mbarriers, with
//     two A and two D buffers, so the three overlap across tiles.
#include <cstdint>
#include <cuda_fp16.h>
#include <type_traits>

#include "common.cuh"
#include "walk_params.cuh"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA0 = 0, kColA1 = 128;  // A buffers; D buffers follow at column 256

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// sm_100 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;            // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both fp16 (fmt 0) or
// both bf16 (fmt 1), both K-major, M = 128, N.
__host__ __device__ constexpr uint32_t f16_idesc(uint32_t fmt, int N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(kTile >> 4) << 24);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(mbar)) : "memory");
}

// One try_wait suspends the thread for up to a hardware-chosen time and returns false
// if the phase has not completed by then. No suspend-time hint: with one, a waiting
// thread took ~200 cycles to resume after the completing arrival, ~125 without.
__device__ __forceinline__ bool mbar_try(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  return done != 0;
}

// Bounded wait for an mbarrier phase; false after timeout_ns of wall-clock time.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try(mbar, parity))
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  return true;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
        "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]),
        "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// The same store from 8 raw 16-byte chunks (bf16 rows need no conversion).
__device__ __forceinline__ void tmem_st32_u4(uint32_t taddr, const uint4 (&c)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};"
      ::"r"(taddr), "r"(c[0].x), "r"(c[0].y), "r"(c[0].z), "r"(c[0].w), "r"(c[1].x), "r"(c[1].y),
        "r"(c[1].z), "r"(c[1].w), "r"(c[2].x), "r"(c[2].y), "r"(c[2].z), "r"(c[2].w), "r"(c[3].x),
        "r"(c[3].y), "r"(c[3].z), "r"(c[3].w), "r"(c[4].x), "r"(c[4].y), "r"(c[4].z), "r"(c[4].w),
        "r"(c[5].x), "r"(c[5].y), "r"(c[5].z), "r"(c[5].w), "r"(c[6].x), "r"(c[6].y), "r"(c[6].z),
        "r"(c[6].w), "r"(c[7].x), "r"(c[7].y), "r"(c[7].z), "r"(c[7].w)
      : "memory");
}

// Loads of tensor-memory columns into registers: x4 / x8 pieces without a wait, then
// one tcgen05.wait::ld for all of them.
__device__ __forceinline__ void tmem_ld4_nowait(uint32_t a, float* d) {
  uint32_t r0, r1, r2, r3;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a) : "memory");
  d[0] = __uint_as_float(r0); d[1] = __uint_as_float(r1); d[2] = __uint_as_float(r2); d[3] = __uint_as_float(r3);
}
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t a, float* d) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]) : "r"(a) : "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) d[j] = __uint_as_float(r[j]);
}
template <int CH>
__device__ __forceinline__ void tmem_ld_cols(uint32_t a, float* d) {
  static_assert(CH == 4 || CH % 8 == 0, "4 or a multiple of 8 columns");
  if constexpr (CH == 4) {
    tmem_ld4_nowait(a, d);
  } else {
#pragma unroll
    for (int c = 0; c < CH; c += 8) tmem_ld8_nowait(a + c, d + c);
  }
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// CH consecutive columns of one accumulator, one wait.
template <int CH>
__device__ __forceinline__ void tmem_ld1(uint32_t a0, float (&d0)[CH]) {
  tmem_ld_cols<CH>(a0, d0);
  tmem_wait_ld();
}
// CH consecutive columns of each of the two K-half accumulators, one wait.
template <int CH>
__device__ __forceinline__ void tmem_ld2(uint32_t a0, uint32_t a1, float (&d0)[CH], float (&d1)[CH]) {
  tmem_ld_cols<CH>(a0, d0);
  tmem_ld_cols<CH>(a1, d1);
  tmem_wait_ld();
}

// Column maxima of NC packed words per lane over the 32 lanes of a warp: plain
// butterfly rounds while the offset is at least NC, then reduce-scatter rounds that
// halve the columns a lane holds; lane l returns the maximum of column l % NC.
template <int NC>
__device__ __forceinline__ uint64_t column_max_scatter(uint64_t (&x)[NC], int lane) {
#pragma unroll
  for (int o = 16; o >= NC; o >>= 1)
#pragma unroll
    for (int k = 0; k < NC; ++k) x[k] = umax64(x[k], __shfl_xor_sync(kFull, x[k], o));
#pragma unroll
  for (int w = NC / 2; w >= 1; w >>= 1) {
    const bool up = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const uint64_t keep = up ? x[k + w] : x[k];
      const uint64_t send = up ? x[k] : x[k + w];
      x[k] = umax64(keep, __shfl_xor_sync(kFull, send, w));
    }
  }
  return x[0];
}

// 4 x 4 transpose inside each group of 4 lanes: on entry lane j holds row j
// (x[c] = a[j][c]); on return it holds column j (x[r] = a[r][j]).
__device__ __forceinline__ void transpose4(float (&x)[4], int lane) {
  const bool odd = lane & 1, hi = lane & 2;
  const float s0 = odd ? x[0] : x[1];
  const float s1 = odd ? x[2] : x[3];
  const float r0 = __shfl_xor_sync(kFull, s0, 1);
  const float r1 = __shfl_xor_sync(kFull, s1, 1);
  if (odd) { x[0] = r0; x[2] = r1; } else { x[1] = r0; x[3] = r1; }
  const float t0 = hi ? x[0] : x[2];
  const float t1 = hi ? x[1] : x[3];
  const float q0 = __shfl_xor_sync(kFull, t0, 2);
  const float q1 = __shfl_xor_sync(kFull, t1, 2);
  if (hi) { x[0] = q0; x[1] = q1; } else { x[2] = q0; x[3] = q1; }
}

// Four int8 codes (one 32-bit word) as two fp16x2 words holding the exact integers.
__device__ __forceinline__ void int8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;  // biased bytes q + 128 in [1, 255]
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(x), "r"(0x64646464u));  // 1024 + byte
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(x), "r"(0x64646464u));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ha);
  hi = *reinterpret_cast<const uint32_t*>(&hb);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_pending(int pending) {
  switch (pending) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
  }
}

}  // namespace

// N = 16, 32 or 64 padded request rows. Warp roles inside the tile pipeline:
//   warps 0-7   producers: quadrant w & 3 (tensor-memory lanes), K half w >> 2; each
//               thread converts half of one W2 row of the tile into tensor memory.
//   warps 8-15  epilogue: quadrant w & 3, column half (w - 8) >> 2; each sums the two
//               K-half accumulators and scores the entries.
//   MMA issue   one thread per K half issues that half's 8 MMAs of a tile into its own
//               accumulator once the half's 4 producer warps are done (two issuing
//               threads double the issue rate): lane 0 of warps 16 and 17, which do
//               nothing else, for N = 16; lane 0 of producer warps 0 and 5 for N = 32
//               and 64, where the epilogue needs every register of a 512-thread CTA.
// Roles hand tiles over through mbarriers (A full/empty per buffer and K half, D
// full/empty per buffer), with two A and two D buffers in tensor memory.
// ROWS (with PROB): per-row modes or temperatures; the other instances score every
// column with the kernel's mode and temperature.
template <bool INT8, bool PROB, bool LOGITS, int N, bool ROWS>
__global__ void __launch_bounds__(walk_tc_threads(N), 1) walk_tc_kernel(const __grid_constant__ WalkParams p) {
  static_assert(PROB || !ROWS, "per-row settings come with sampled rows");
  constexpr bool kOwnIssuers = walk_tc_threads(N) > kWalkThreads;  // warps 16, 17 issue the MMAs
  constexpr int kWarps = walk_tc_threads(N) / 32;
  constexpr int NC = N / 2;                          // columns per epilogue warp
  constexpr int kRowBytes = INT8 ? kRank : 2 * kRank;
  constexpr int kChunks = kRowBytes / 16;            // 16-byte chunks per W2 row
  constexpr int kHalfChunks = kChunks / 2;           // per producer thread and tile
  constexpr int kPassChunks = INT8 ? 4 : 8;          // chunks per 32-column store
  constexpr uint32_t kIdesc = f16_idesc(INT8 ? 0u : 1u, N);
  constexpr uint32_t kColD = 256;                    // D buffers from column 256
  // N = 64: one accumulator per D buffer, K half 1 issued after K half 0 (ordered by
  // an mbarrier between the two issuing threads) onto half 0's partial sums, so the
  // epilogue loads and adds nothing twice; smaller N: one accumulator per K half at
  // kColD + (2 buf + half) N, the two halves issued concurrently.
  constexpr bool kOneAcc = N == 64;
  // N = 64 with scores through bf16 or draft_logits (the heavier register load):
  // column maxima reduced through shared memory instead of lane shuffles
  constexpr bool kSmemReduce = N == 64 && (PROB || LOGITS);

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start, by an offset from smem_raw so that every derived pointer
  // stays a shared-memory pointer (32-bit shared loads and stores)
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* b_s = smem;                                      // N x 512 bytes
  uint16_t* base_stage = reinterpret_cast<uint16_t*>(b_s + N * 512);  // [8 warps][2][N/2][32]
  unsigned char* w2s = b_s + N * 512 + walk_tc_stage_bytes(N);      // resident rows
  float* scale_s = reinterpret_cast<float*>(w2s + static_cast<size_t>(p.resident_rows) * kRowBytes);
  int* prev_s = reinterpret_cast<int*>(scale_s + (INT8 ? p.slice_cap : 0));   // [64]
  uint64_t* seed_s = reinterpret_cast<uint64_t*>(prev_s + 64);    // [64] per-request seeds
  uint64_t* best_s = seed_s + 64;
  uint64_t* red_s = best_s + 64;                                  // [4][64]
  float2* inv_s = reinterpret_cast<float2*>(red_s + 4 * 64);       // 2^-s as two factors
  float* invT_s = reinterpret_cast<float*>(inv_s + 2);            // [64] 1/T per row (fp32)
  uint64_t* gmask_s = reinterpret_cast<uint64_t*>(invT_s + 64);   // bit b: row b greedy
  uint64_t* mbar = gmask_s + 1;                                    // [30]
  uint64_t* a_full = mbar;        // [buf * 2 + half], 4 arrivals
  uint64_t* a_empty = mbar + 4;   // [buf * 2 + half], 1 commit
  uint64_t* d_full = mbar + 8;    // [buf], 2 commits
  uint64_t* d_empty = mbar + 10;  // [buf], 8 arrivals
  uint64_t* s_full = mbar + 12;   // [epilogue warp * 2 + stage buffer], 1 arrival + bytes
  uint64_t* h0_done = mbar + 28;  // [buf], one accumulator: K half 0 of the tile issued
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(mbar + 30);
  int* flag = reinterpret_cast<int*>(tbase_s + 1);
  int* sh_amax = flag + 1;        // largest finite |e| of the batch, as fp32 bits

  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t v0 = slice_start(cta, G, p.V), v1 = slice_start(cta + 1, G, p.V);
  const int n = static_cast<int>(v1 - v0);
  const int res = min(p.resident_rows, n);
  const int T = (n + kTile - 1) / kTile;
  const unsigned char* w2g = (INT8 ? reinterpret_cast<const unsigned char*>(p.w2q)
                                   : reinterpret_cast<const unsigned char*>(p.w2)) +
                             static_cast<size_t>(v0) * kRowBytes;
  const bool skip0 = (p.sync.flags & DSPARK_FLAG_SKIP_ARRIVAL_CTA0) && cta == 0;
  const bool producer = warp < 8;
  const int q = warp & 3;                                          // tensor-memory lane quadrant
  // producers and issuers: K half; epilogue: column half
  const int half = (kOwnIssuers && warp >= 16) ? warp - 16 : (warp >> 2) & 1;
  // MMA issuers: producer warp 0 (K half 0) and 5 (K half 1), on different SM sub-partitions
  const bool issuer = kOwnIssuers ? warp >= 16 : (producer && q == half);

  // ---- set-up: zero B, scales, previous tokens, barriers, tensor memory
  for (int t = tid; t < N * 512 / 16; t += blockDim.x) reinterpret_cast<uint4*>(b_s)[t] = make_uint4(0, 0, 0, 0);
  if (INT8)
    for (int r = tid; r < n; r += blockDim.x) scale_s[r] = __ldg(p.scales + v0 + r);
  for (int t = tid; t < 64; t += blockDim.x) {
    const bool sampled = t < p.bs && row_sampled(p, PROB, t);
    seed_s[t] = sampled ? p.seeds[t] : 0ull;
    // 1/T rounded to fp32 from the double quotient, as the host does for the scalar T
    if constexpr (ROWS) invT_s[t] = sampled ? static_cast<float>(1.0 / static_cast<double>(row_temperature(p, t))) : 1.0f;
  }
  for (int t = tid; t < p.bs; t += blockDim.x) {
    const int32_t tok = p.prev[t];
    const bool okt = tok >= 0 && static_cast<int64_t>(tok) < p.V;
    const bool settings = row_settings_ok(p, PROB, t);
    prev_s[t] = okt && settings ? tok : -1;
    if (!okt && cta == 0) report(p.sync.status_dev, DSPARK_ERR_BAD_TOKEN);
    if (!settings && cta == 0) report(p.sync.status_dev, DSPARK_ERR_INVALID_ARG);
  }
  if (tid == 0) {
    const uint32_t counts[12] = {4, 4, 4, 4, 1, 1, 1, 1, 2, 2, 8, 8};
    for (int b = 0; b < 30; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&mbar[b])), "r"(b < 12 ? counts[b] : 1u));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *sh_amax = 0;
    if constexpr (ROWS) {
      uint64_t gm = 0ull;
      for (int b = 0; b < p.bs; ++b)
        if (!row_sampled(p, PROB, b)) gm |= 1ull << b;
      *gmask_s = gm;
    }
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tbase_s)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  prefetch_base_slice(p, v0, n, 0);
  prefetch_base_slice(p, v0, n, 1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase_s;
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  bool ok = true;
  int g_base = 0;        // tiles processed by all earlier positions (buffer / phase bookkeeping)
  int last_issued = -1;  // issuers: last tile whose MMAs were committed
  uint32_t stage_ph = 0;  // epilogue: bit b = parity of stage buffer b's next completion

  for (int i = 0; i < p.K && ok; ++i) {
    // ---- B operand: the embedding rows of this position's previous tokens
    // (at most 4 rows per warp: issue every load before converting any row)
    uint4 wrow[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int b = warp + kWarps * r;
      const int tok = b < p.bs ? prev_s[b] : -1;
      wrow[r] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(tok) * kRank) + lane)
                         : make_uint4(0, 0, 0, 0);
    }
    // int8 W2: one power-of-two scale 2^s for the whole batch, with the largest finite
    // |e| of all rows in [2^14, 2^15) after scaling.
    int shift = 0;
    if constexpr (INT8) {
      float amax = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int b = warp + kWarps * r;
        if (b >= p.bs) break;
        const uint32_t ww[4] = {wrow[r].x, wrow[r].y, wrow[r].z, wrow[r].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float lo = bf16_lo(ww[t]), hi = bf16_hi(ww[t]);
          if (isfinite(lo)) amax = fmaxf(amax, fabsf(lo));
          if (isfinite(hi)) amax = fmaxf(amax, fabsf(hi));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      if (lane == 0 && amax > 0.f) atomicMax(sh_amax, __float_as_int(amax));
      __syncthreads();
      const float am = __int_as_float(*reinterpret_cast<volatile int*>(sh_amax));
      if (am > 0.f) {
        int ex;
        frexpf(am, &ex);  // am = f 2^ex, f in [0.5, 1)
        shift = 15 - ex;  // am 2^shift in [2^14, 2^15)
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int b = warp + kWarps * r;
      if (b >= p.bs) break;
      uint4 w = wrow[r];
      if constexpr (INT8) {
        const float s_lo = __int_as_float((shift / 2 + 127) << 23);
        const float s_hi = __int_as_float((shift - shift / 2 + 127) << 23);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t h[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = __fmul_rn(__fmul_rn(bf16_lo(ww[t]), s_lo), s_hi);
          const float c = __fmul_rn(__fmul_rn(bf16_hi(ww[t]), s_lo), s_hi);
          const __half2 hh = __floats2half2_rn(a, c);
          h[t] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        w = make_uint4(h[0], h[1], h[2], h[3]);
      }
      const int kb = lane >> 3, ch = lane & 7;
      *reinterpret_cast<uint4*>(b_s + kb * N * 128 + b * 128 + ((ch ^ (b & 7)) * 16)) = w;
    }
    if (tid == 0)
      *inv_s = make_float2(__int_as_float(((-shift) / 2 + 127) << 23),
                           __int_as_float(((-shift) - (-shift) / 2 + 127) << 23));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();  // B written and visible to the tensor core; 2^-s published
    if (tid == 0) *sh_amax = 0;  // every thread read it before the barrier

    bool failed = false;
    // This K half's 8 MMAs of tile g into D buffer buf (the caller has waited for A,
    // the D buffer and, with one accumulator, for K half 0), then the commits.
    auto issue_half = [&](int buf, int g) {
      tc_fence_after();
      const uint32_t a_col = buf ? kColA1 : kColA0;
      const uint32_t d_col = kColD + (kOneAcc ? buf * N : (2 * buf + half) * N);
      const uint32_t b_base = smem_u32(b_s);
      const uint32_t acc0 = (kOneAcc && half == 1) ? 1u : 0u;  // half 1 adds onto half 0
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) {
        const int kk = 8 * half + k8;
        const uint64_t bd = sw128_desc(b_base + (kk / 4) * N * 128 + (kk % 4) * 32);
        mma_f16(tmem + d_col, tmem + a_col + 8 * kk, bd, kIdesc, k8 > 0 ? 1u : acc0);
      }
      mma_commit(&d_full[buf]);
      mma_commit(&a_empty[buf * 2 + half]);
      if (kOneAcc && half == 0) {
        // K half 1's MMAs are issued after all of these (tensor-core operations ordered
        // across threads through the fence and the mbarrier): a fixed summation order,
        // so the walk is deterministic
        tc_fence_before();
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&h0_done[buf])) : "memory");
      }
      last_issued = g;
    };
    if (producer) {
      // ---------------------------------------------------------------- producers
      const bool fill_now = (i == 0);
      int n_res_tiles = 0;
      if (fill_now) {  // position 0: resident rows arrive through cp.async, a group per tile
        for (int t = 0; t < T && t * kTile < res; ++t) {
          const int rr = t * kTile + 32 * q + lane;
          if (rr < res) {
#pragma unroll
            for (int j = 0; j < kHalfChunks; ++j) {
              const int ch = kHalfChunks * half + j;
              const int pos = ch ^ (rr & (kChunks - 1));
              cp_async16(w2s + static_cast<size_t>(rr) * kRowBytes + 16 * pos,
                         w2g + static_cast<size_t>(rr) * kRowBytes + 16 * ch);
            }
          }
          cp_async_commit();
          ++n_res_tiles;
        }
      }
      // This thread's half row of tile t: kHalfChunks 16-byte chunks, loaded as passes
      // of kPassChunks (one 32-column tensor-memory store each).
      auto load_pass = [&](int t, int pass, uint4 (&c)[kPassChunks]) {
        const int rr = t * kTile + 32 * q + lane;
        const int ch0 = kHalfChunks * half + kPassChunks * pass;
        if (rr < res) {  // resident row: shared memory, XOR-swizzled chunks
          const uint4* row = reinterpret_cast<const uint4*>(w2s + rr * kRowBytes);
#pragma unroll
          for (int j = 0; j < kPassChunks; ++j) c[j] = row[(ch0 + j) ^ (rr & (kChunks - 1))];
        } else if (rr < n) {  // streamed row: L2
          const uint4* row = reinterpret_cast<const uint4*>(w2g + static_cast<size_t>(rr) * kRowBytes) + ch0;
#pragma unroll
          for (int j = 0; j < kPassChunks; ++j) c[j] = __ldg(row + j);
        } else {
#pragma unroll
          for (int j = 0; j < kPassChunks; ++j) c[j] = make_uint4(0, 0, 0, 0);
        }
      };
      auto store_pass = [&](const uint4 (&c)[kPassChunks], uint32_t col) {
        if constexpr (INT8) {
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            int8x4_to_f16x4(c[j].x, v[8 * j + 0], v[8 * j + 1]);
            int8x4_to_f16x4(c[j].y, v[8 * j + 2], v[8 * j + 3]);
            int8x4_to_f16x4(c[j].z, v[8 * j + 4], v[8 * j + 5]);
            int8x4_to_f16x4(c[j].w, v[8 * j + 6], v[8 * j + 7]);
          }
          tmem_st32(tmem + lane_off + col, v);
        } else {
          tmem_st32_u4(tmem + lane_off + col, c);
        }
      };
      // int8: both passes of the next tile are prefetched; bf16 (twice the bytes): the
      // first pass is prefetched and the second loaded just before its store.
      uint4 c0[kPassChunks], c1[kPassChunks];
      if (T > 0) {
        if (fill_now && n_res_tiles > 0) cp_async_wait_pending(n_res_tiles - 1);
        load_pass(0, 0, c0);
        if constexpr (INT8) load_pass(0, 1, c1);
      }
      for (int t = 0; t < T; ++t) {
        const int g = g_base + t, buf = g & 1, u = g >> 1;
        if (u >= 1 && !mbar_wait(&a_empty[buf * 2 + half], (u - 1) & 1, p.sync.timeout_ns)) failed = true;
        if (__shfl_sync(kFull, failed ? 1 : 0, 0)) { failed = true; break; }
        tc_fence_after();
        const uint32_t acol = (buf ? kColA1 : kColA0) + 64 * half;
        store_pass(c0, acol);
        if constexpr (!INT8) load_pass(t, 1, c1);
        store_pass(c1, acol + 32);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&a_full[buf * 2 + half])) : "memory");
        if (!kOwnIssuers && issuer && lane == 0) {
          // MMA issue for this K half: A complete (all 4 quadrants), D buffer free.
          bool good = mbar_wait(&a_full[buf * 2 + half], u & 1, p.sync.timeout_ns);
          if (good && u >= 1) good = mbar_wait(&d_empty[buf], (u - 1) & 1, p.sync.timeout_ns);
          if (kOneAcc && good && half == 1) good = mbar_wait(&h0_done[buf], u & 1, p.sync.timeout_ns);
          if (!good) {
            failed = true;
          } else {
            issue_half(buf, g);
          }
        }
        if (t + 1 < T) {  // next tile's data in flight while this warp waits (issuers: after the MMAs)
          if (fill_now && t + 1 < n_res_tiles) cp_async_wait_pending(n_res_tiles - 2 - t);
          load_pass(t + 1, 0, c0);
          if constexpr (INT8) load_pass(t + 1, 1, c1);
        }
        if (__shfl_sync(kFull, failed ? 1 : 0, 0)) { failed = true; break; }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (kOwnIssuers && issuer) {
      // ------------------------------------------------------------- MMA issue
      // Lane 0 issues this K half's 8 MMAs of every tile into its own accumulator once
      // the 4 producer warps of the half have stored the tile and the epilogue has
      // released the D buffer.
      if (lane == 0) {
        for (int t = 0; t < T; ++t) {
          const int g = g_base + t, buf = g & 1, u = g >> 1;
          bool good = mbar_wait(&a_full[buf * 2 + half], u & 1, p.sync.timeout_ns);
          if (good && u >= 1) good = mbar_wait(&d_empty[buf], (u - 1) & 1, p.sync.timeout_ns);
          if (kOneAcc && good && half == 1) good = mbar_wait(&h0_done[buf], u & 1, p.sync.timeout_ns);
          if (!good) { failed = true; break; }
          issue_half(buf, g);
        }
      }
      __syncwarp();
    } else {
      // -------------------------------------------------------------- epilogue
      // Thread = tensor-memory lane = vocabulary row 32 q + lane of the tile; the
      // warp's NC columns (request rows) are warp-uniform. Each thread keeps, per
      // column, the running maximum of its rows over the tiles (max.NaN: a NaN sticks)
      // and the tile where it was first reached: the tile is rewritten when the maximum
      // changes (an unordered compare, so the first NaN counts) unless it already is
      // NaN. Equal values (also -0 and +0) never rewrite it, so the first maximum stays.
      // Tiles are 8-bit fields, four columns per register. The lanes and quadrants are
      // combined once per position. The base logits of the warp's rows and columns are
      // staged in shared memory one tile ahead.
      // columns per accumulator load: as many as the registers allow (one accumulator at
      // N = 64 leaves room for twice as many)
      constexpr int CHG = NC < 8 ? NC : (kOneAcc ? (PROB ? 8 : 16) : (PROB ? 4 : 8));
      static_assert(NC % CHG == 0, "the column chunks must tile the warp's columns");
      static_assert(!PROB || CHG % 4 == 0, "Philox blocks are drawn for groups of 4 columns");
      const int cb = half * NC;                                 // first column of the warp
      const int ncol = max(0, min(NC, p.bs - cb));              // live columns (uniform)
      const int ew = warp - 8;
      [[maybe_unused]] const uint32_t wg = ROWS ? static_cast<uint32_t>(*gmask_s >> cb) : 0u;  // greedy columns
      uint16_t* stage_s = base_stage + static_cast<size_t>(ew) * 2 * NC * 32;  // [2][NC][32]
      // request rows whose previous token was out of range are skipped
      const uint32_t live = __ballot_sync(kFull, lane < ncol && prev_s[cb + min(lane, NC - 1)] >= 0);
      const size_t bstride = static_cast<size_t>(p.K) * static_cast<size_t>(p.V);
      const uint16_t* brow = p.base + static_cast<size_t>(i) * p.V + v0;  // + b K V + row
      // Base logits of tile t into stage buffer t & 1: one tensor-map tile copy (box of
      // 32 rows x 1 position x NC requests, completion counted in bytes on s_full) when
      // the host could describe base, else 16-byte cp.async pieces of 8 rows (slices
      // start on multiples of 32 rows and, with V a multiple of 8, end on multiples of
      // 8, so a piece is entirely inside or outside), else plain loads.
      const bool tma = p.base_tma != 0;
      // logits through the stage buffer only when the base arrives by tensor-map copy too
      [[maybe_unused]] const bool ltma = tma && p.logits_tma != 0;
      const bool vec_ok = (p.V & 7) == 0 && (reinterpret_cast<uintptr_t>(p.base) & 15u) == 0;
      uint64_t* sfull = s_full + 2 * (warp - 8);
      int staged = -1;       // last tile whose copy was issued
      int landed = -1;       // last tile whose copy was waited for
      auto stage = [&](int t) {
        const int sb = t & 1;
        const int r0 = t * kTile + 32 * q;
        uint16_t* buf_s = stage_s + sb * NC * 32;
        if (tma) {
          if (lane == 0) {
            constexpr uint32_t kBytes = NC * 32 * 2;
            if (LOGITS && ltma) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         ::"r"(smem_u32(&sfull[sb])), "r"(kBytes) : "memory");
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3, %4}], [%5];"
                ::"r"(smem_u32(buf_s)), "l"(reinterpret_cast<uint64_t>(&p.base_map)),
                  "r"(static_cast<int>(v0) + r0), "r"(i), "r"(cb), "r"(smem_u32(&sfull[sb]))
                : "memory");
          }
        } else {
          for (int e = lane; e < ncol * 4; e += 32) {
            const int j = e >> 2, c8 = e & 3;
            if (!((live >> j) & 1u)) continue;
            const int rr = r0 + 8 * c8;
            uint16_t* dst = buf_s + j * 32 + 8 * c8;
            const uint16_t* src = brow + static_cast<size_t>(cb + j) * bstride + rr;
            if (vec_ok) {
              if (rr < n) cp_async16(dst, src);
            } else {
#pragma unroll
              for (int e8 = 0; e8 < 8; ++e8) dst[e8] = rr + e8 < n ? src[e8] : 0;
            }
          }
          cp_async_commit();
        }
        staged = t;
      };
      // Wait until tile t's copy has landed (bounded); true on success.
      auto land = [&](int t) -> bool {
        bool good = true;
        if (tma) {
          const int sb = t & 1;
          good = mbar_wait(&sfull[sb], (stage_ph >> sb) & 1u, p.sync.timeout_ns);
          stage_ph ^= 1u << sb;
        } else {
          cp_async_wait_pending(staged > t ? 1 : 0);
        }
        landed = t;
        return good;
      };
      float bv[NC];
      uint32_t bt[(NC + 3) / 4];
#pragma unroll
      for (int j = 0; j < NC; ++j) bv[j] = -INFINITY;
#pragma unroll
      for (int w = 0; w < (NC + 3) / 4; ++w) bt[w] = 0u;
      if (T > 0) stage(0);
      const float2 inv = inv_s[0];
      // One tile; FULL: every row of the tile lies in the slice.
      auto tile = [&](auto full_tag, int t, int buf) {
        constexpr bool FULL = decltype(full_tag)::value;
        const int rr = t * kTile + 32 * q + lane;
        const bool valid = rr < n;
        [[maybe_unused]] float c = 1.f;
        if constexpr (INT8) c = __fmul_rn(__fmul_rn(valid ? scale_s[rr] : 0.f, inv.x), inv.y);
        const uint32_t trep = static_cast<uint32_t>(t) * 0x01010101u;
        const uint16_t* bsm = stage_s + (t & 1) * NC * 32 + lane;
        [[maybe_unused]] uint16_t* bsw = stage_s + (t & 1) * NC * 32 + lane;
#pragma unroll
        for (int cc = 0; cc < NC / CHG; ++cc) {
          if (cc * CHG >= ncol) break;
          float dsum[CHG];  // the contraction D of the thread's row, the chunk's columns
          if constexpr (kOneAcc) {
            tmem_ld1<CHG>(tmem + lane_off + kColD + buf * N + cb + cc * CHG, dsum);
          } else {
            float d1[CHG];
            const uint32_t dcol = kColD + 2 * buf * N + cb + cc * CHG;
            tmem_ld2<CHG>(tmem + lane_off + dcol, tmem + lane_off + dcol + N, dsum, d1);
#pragma unroll
            for (int k = 0; k < CHG; ++k) dsum[k] = __fadd_rn(dsum[k], d1[k]);
          }
          float sc[CHG];  // scores of this thread's row in the chunk's columns
#pragma unroll
          for (int k = 0; k < CHG; ++k) {
            const int j = cc * CHG + k;  // columns past bs or of dead rows are computed and discarded
            const float bvl = __uint_as_float(static_cast<uint32_t>(bsm[j * 32]) << 16);
            float l;
            if constexpr (INT8) l = __fmaf_rn(dsum[k], c, bvl);
            else l = __fadd_rn(dsum[k], bvl);
            if constexpr (!FULL) l = valid ? l : -INFINITY;
            [[maybe_unused]] const uint16_t lh = f32_to_bf16_bits(l);
            if constexpr (LOGITS) {
              if (ltma) bsw[j * 32] = lh;  // the tile of logits replaces the tile of base
              else if (valid && j < ncol)
                p.logits[static_cast<size_t>(cb + j) * bstride + static_cast<size_t>(i) * p.V + v0 + rr] = lh;
            }
            if constexpr (PROB) {
              const float lb = bf16_to_f32(lh);
              if constexpr (ROWS)  // greedy rows of a mixed batch score the fp32 logit
                sc[k] = ((wg >> j) & 1u) ? l : __fmul_rn(lb, invT_s[cb + j]);
              else  // 1/T = 1 multiplies exactly
                sc[k] = __fmul_rn(lb, p.inv_temperature);
            } else {
              sc[k] = l;
            }
          }
          if constexpr (PROB) {
            // Gumbel noise: lane 4m + k draws the Philox block of rows 4m..4m+3 (of
            // this warp's 32) and column jb + k, then a 4 x 4 transpose inside the lane
            // quad leaves every lane the draws of its own row for columns jb..jb+3.
            const uint32_t m = (static_cast<uint32_t>(v0) + t * kTile + 32 * q) / 4 + (lane >> 2);
#pragma unroll
            for (int h4 = 0; h4 < CHG / 4; ++h4) {
              const int bq = cb + cc * CHG + 4 * h4 + (lane & 3);
              const uint4 w = philox_block(seed_s[bq], bq, i, m);
              float g4[4] = {gumbel_from_word(w.x), gumbel_from_word(w.y), gumbel_from_word(w.z),
                             gumbel_from_word(w.w)};
              transpose4(g4, lane);
#pragma unroll
              for (int r = 0; r < 4; ++r)
                if (!ROWS || !((wg >> (cc * CHG + 4 * h4 + r)) & 1u)) sc[4 * h4 + r] = __fadd_rn(sc[4 * h4 + r], g4[r]);
            }
          }
#pragma unroll
          for (int k = 0; k < CHG; ++k) {
            const int j = cc * CHG + k;
            float nv;
            asm("max.NaN.f32 %0, %1, %2;" : "=f"(nv) : "f"(bv[j]), "f"(sc[k]));
            asm("{ .reg .pred r, u; setp.num.f32 r, %1, %1; setp.neu.and.f32 u, %2, %1, r; "
                "@u lop3.b32 %0, %0, %3, %4, 0xB8; }"
                : "+r"(bt[j >> 2]) : "f"(bv[j]), "f"(nv), "r"(0xFFu << (8 * (j & 3))), "r"(trep));
            bv[j] = nv;
          }
        }
      };
      for (int t = 0; t < T; ++t) {
        const int g = g_base + t, buf = g & 1, u = g >> 1;
        if (t + 1 < T) stage(t + 1);
        if (!mbar_wait(&d_full[buf], u & 1, p.sync.timeout_ns)) failed = true;
        if (!failed && !land(t)) failed = true;
        if (__shfl_sync(kFull, failed ? 1 : 0, 0)) { failed = true; break; }
        tc_fence_after();
        __syncwarp();
        if ((t + 1) * kTile <= n) tile(std::true_type{}, t, buf);
        else tile(std::false_type{}, t, buf);
        tc_fence_before();
        __syncwarp();
        if constexpr (LOGITS) {
          // the warp's 32 rows of logits, unless they all lie past the slice (rows past
          // V and requests past bs are clipped by the copy)
          if (ltma && lane == 0 && t * kTile + 32 * q < n) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile(
                "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                ::"l"(reinterpret_cast<uint64_t>(&p.logits_map)), "r"(static_cast<int>(v0) + t * kTile + 32 * q),
                  "r"(i), "r"(cb), "r"(smem_u32(stage_s + (t & 1) * NC * 32))
                : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
        }
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&d_empty[buf])) : "memory");
      }
      // copies still in flight after a failure land before the CTA can leave; logits
      // stores are complete before the position ends
      for (int t = landed + 1; t <= staged; ++t) land(t);
      if (LOGITS && ltma && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      asm volatile("cp.async.wait_all;" ::: "memory");
      // per column: (orderable key, first index) maximum over the warp's 32 rows
      if constexpr (NC <= 8) {
        // few columns: one warp-wide integer max of the keys per column; the first
        // index among the lanes that reach it is the smallest (tile, lane)
#pragma unroll
        for (int j = 0; j < NC; ++j) {
          if (j >= ncol) break;
          const uint32_t key = order_key(bv[j]);
          const uint32_t kmax = __reduce_max_sync(kFull, key);
          const uint32_t cand = __ballot_sync(kFull, key == kmax);
          const uint32_t tj = (bt[j >> 2] >> (8 * (j & 3))) & 0xFFu;
          uint32_t pos = key == kmax ? ((tj << 5) | static_cast<uint32_t>(lane)) : 0xFFFFFFFFu;
          if (__popc(cand) > 1) pos = __reduce_min_sync(kFull, pos);
          else pos = __shfl_sync(kFull, pos, __ffs(cand) - 1);
          if (lane == 0)
            red_s[q * 64 + cb + j] =
                pack_best(kmax, static_cast<uint32_t>(v0) + 32u * q + (pos & 31u) + (pos >> 5) * kTile);
        }
      } else if constexpr (kSmemReduce) {
        // packed words transposed through the warp's stage buffer (idle now), in two
        // rounds of RW = NC / 2 columns: lane l writes its RW words as row l ([32][RW],
        // word k at slot k ^ (l % RW)); lane g RW + k then takes the maximum of column
        // k over rows g RW .. g RW + RW - 1, and the 32 / RW row groups are combined by
        // butterflies.
        __syncwarp();
        constexpr int RW = NC / 2;
        static_assert((RW & (RW - 1)) == 0 && RW >= 8 && RW <= 16, "transpose rounds of 8 or 16 columns");
        uint64_t* tr = reinterpret_cast<uint64_t*>(stage_s);  // 32 x RW words: the 2 x NC x 32 stage
        const uint32_t vlane = static_cast<uint32_t>(v0) + 32u * q + lane;
        const int kc = lane & (RW - 1), gr = lane / RW;
#pragma unroll
        for (int r0 = 0; r0 < NC; r0 += RW) {
#pragma unroll
          for (int k = 0; k < RW; ++k) {
            const int j = r0 + k;
            const uint32_t tj = (bt[j >> 2] >> (8 * (j & 3))) & 0xFFu;
            tr[lane * RW + (k ^ (lane & (RW - 1)))] = j < ncol ? pack_best(order_key(bv[j]), vlane + tj * kTile) : 0ull;
          }
          __syncwarp();
          uint64_t m = 0ull;
#pragma unroll
          for (int rr = 0; rr < RW; ++rr) m = umax64(m, tr[(gr * RW + rr) * RW + (kc ^ rr)]);
#pragma unroll
          for (int o = RW; o < 32; o <<= 1) m = umax64(m, __shfl_xor_sync(kFull, m, o));
          if (lane < RW && r0 + lane < ncol) red_s[q * 64 + cb + r0 + lane] = m;
          __syncwarp();
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before the next tensor-map copies
      } else {
        // many columns: packed words, reduce-scattered across the lanes
        const uint32_t vlane = static_cast<uint32_t>(v0) + 32u * q + lane;
        constexpr int RG = NC < 16 ? NC : 16;  // columns per reduction group (register budget)
        static_assert(NC % RG == 0 && (RG & (RG - 1)) == 0, "reduction groups: a power of two tiling NC");
#pragma unroll
        for (int g0 = 0; g0 < NC; g0 += RG) {
          uint64_t x[RG];
#pragma unroll
          for (int k = 0; k < RG; ++k) {
            const int j = g0 + k;
            const uint32_t tj = (bt[j >> 2] >> (8 * (j & 3))) & 0xFFu;
            x[k] = j < ncol ? pack_best(order_key(bv[j]), vlane + tj * kTile) : 0ull;
          }
          const uint64_t xm = column_max_scatter<RG>(x, lane);
          if (lane < RG && g0 + lane < ncol) red_s[q * 64 + cb + g0 + lane] = xm;
        }
      }
    }
    g_base += T;
    if (__syncthreads_or(failed)) {
      // Report, then let the issued MMAs finish (bounded) before tensor memory goes.
      if (tid == 0) give_up(p.sync);
      if (issuer && lane == 0 && last_issued >= 0)
        mbar_wait(&a_empty[(last_issued & 1) * 2 + half], (last_issued >> 1) & 1, p.sync.timeout_ns);
      ok = false;
      break;
    }

    if (tid < p.bs) {
      uint64_t x = umax64(umax64(red_s[tid], red_s[64 + tid]), umax64(red_s[128 + tid], red_s[192 + tid]));
      if (prev_s[tid] < 0) x = 0ull;
      best_s[tid] = x;
      if (x != 0ull && i + 1 < p.K) {
        const uint16_t* row = p.w1 + static_cast<size_t>(unpack_idx(x)) * kRank;
#pragma unroll
        for (int l4 = 0; l4 < 4; ++l4) prefetch_l2(row + 64 * l4);
      }
    }
    if (!exchange_best(p.sync, i, p.bs, skip0 && i == 0, best_s, flag)) { ok = false; break; }
    for (int t = tid; t < p.bs; t += blockDim.x) {
      const int tok = prev_s[t] >= 0 ? unpack_idx(best_s[t]) : -1;
      prev_s[t] = tok;
      if (cta == 0) p.tokens[static_cast<size_t>(t) * p.K + i] = tok;
    }
    reset_behind(p.sync, i, p.bs);
    if (i + 2 < p.K) prefetch_base_slice(p, v0, n, i + 2);
    __syncthreads();
  }

  // ---- release tensor memory (every MMA has completed or the bounded wait gave up)
  asm volatile("cp.async.wait_all;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  if (ok) finish_walk(p.sync, p.K, p.bs, flag);
}

const void* walk_tc_kernel_ptr(bool int8, bool prob, bool logits, int nq, bool rows) {
#define DSPARK_TC(I, P, L, R)                                                  \
  if (int8 == I && prob == P && logits == L && rows == R) {                    \
    if (nq == 4) return (const void*)walk_tc_kernel<I, P, L, 16, R>;           \
    if (nq == 8) return (const void*)walk_tc_kernel<I, P, L, 32, R>;           \
    return (const void*)walk_tc_kernel<I, P, L, 64, R>;                        \
  }
  DSPARK_TC(true, false, false, false)
  DSPARK_TC(true, false, true, false)
  DSPARK_TC(true, true, false, false)
  DSPARK_TC(true, true, true, false)
  DSPARK_TC(true, true, false, true)
  DSPARK_TC(true, true, true, true)
  DSPARK_TC(false, false, false, false)
  DSPARK_TC(false, false, true, false)
  DSPARK_TC(false, true, false, false)
  DSPARK_TC(false, true, true, false)
  DSPARK_TC(false, true, false, true)
  DSPARK_TC(false, true, true, true)
#undef DSPARK_TC
  return nullptr;
}

}  // namespace dspark
