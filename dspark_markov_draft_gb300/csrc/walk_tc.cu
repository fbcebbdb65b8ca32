// Full-vocabulary Markov draft walk with the bias contraction on the 5th-generation
// tensor cores (tcgen05), for batches where W2 . E[256 x bs] is a real dense GEMM.
// Same method and per-position exchange as the CUDA-core walk (vLLM PR #62958,
// "Overview": one cooperative kernel for the whole walk, W2 on chip where it fits,
// one packed atomic per step for the cross-CTA argmax).
//
// One CTA per SM owns a contiguous vocabulary slice, cut into tiles of 128 rows; each
// tile is four 32-row blocks. The slice's last blocks stay resident in shared memory for
// the whole walk (copied once by tensor-map copies with the 128-byte swizzle); its first
// blocks are re-read from L2 at every position, so that they come first in each position
// and their load latency falls in the window of the grid exchange, when the tensor
// cores wait for the next tokens anyway.
//
// Warp roles (24 warps; setmaxnreg moves registers from the producers and the issue
// warps to the epilogue, a split checked on the host against the launch's registers):
//   * warps 0-3, producers: warp q fills tensor-memory lanes 32q..32q+31 of each tile's
//     A operand; a thread converts one W2 row (int8 codes become exact fp16 integers
//     through a byte permute with 0x64 exponent bytes and one packed subtract; bf16 rows
//     are copied). Streamed rows are read from L2 with an evict-last hint, resident rows
//     from the swizzled shared-memory copy. A does not depend on the tokens, so the
//     producers run ahead across positions, limited only by the three A buffers.
//   * warps 4-19, epilogue: warp 4 + 4c + q reads tensor-memory lanes 32q.. (warp % 4 ==
//     q) and the N/4 request columns of column group c. Thread = one vocabulary row of
//     the tile: it adds the base logit (from the staged copy of the tile) to
//     scale_v 2^-s D, scores the entry (greedy: l; probabilistic: bf16(l)/T plus Gumbel
//     noise whose Philox blocks are drawn once per lane quad and exchanged by a 4 x 4
//     transpose), and keeps per column the running maximum and the tile where it was
//     first reached. At the end of a position the same warps reduce the columns, run
//     the grid exchange, gather the next embeddings and build the next B operand.
//   * warps 20 and 21, MMA issue: they take alternate tiles; lane 0 issues the 16 MMAs
//     (M = 128, N, K = 16, A in tensor memory, B in shared memory) of a tile into one of
//     the D buffers, in K order.
//   * warp 22, base-logit copies: tensor-map copies of each tile's base logits for all
//     request columns into a ring of stages, running ahead of the epilogue across
//     positions (the next position's boxes are prefetched to L2).
// Producers, issuers, copier and epilogue hand tiles over through mbarriers (three A
// buffers, two or four D buffers, the base stages, one B-ready barrier per position).
// Every wait is bounded by wall-clock time and watches a CTA fail flag, so a timeout
// anywhere ends every role.
#include <cstdint>
#include <cuda_fp16.h>
#include <type_traits>

#include "common.cuh"
#include "walk_params.cuh"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kABufs = 3;         // A buffers at tensor-memory columns 0, 128, 256
constexpr uint32_t kColD = 384;  // D buffers in the last 128 columns
// D buffers of N columns in the last 128 columns, at most 4
__host__ __device__ constexpr int tc_dbufs(int N) { return N >= 64 ? 2 : 4; }
constexpr int kEpiThreads = kTcEpilogueWarps * 32;
constexpr int kIssuerWarp = kTcProducerWarps + kTcEpilogueWarps;
constexpr int kBarEpi = 1;       // named barrier of the epilogue warps

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

// MMA and commit executed by a whole warp and carried out by one lane only (a predicate
// inside the instruction): the warp's lanes never wait for one another.
__device__ __forceinline__ void mma_f16_if(bool leader, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0; "
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(static_cast<uint32_t>(leader))
      : "memory");
}
__device__ __forceinline__ void mma_commit_if(bool leader, uint64_t* mbar) {
  asm volatile(
      "{ .reg .pred q; setp.ne.b32 q, %1, 0; "
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
      ::"r"(smem_u32(mbar)), "r"(static_cast<uint32_t>(leader)) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(mbar)) : "memory");
}

// One try_wait suspends the thread for up to a hardware-chosen time and returns false
// if the phase has not completed by then (no suspend-time hint: faster wake-up).
__device__ __forceinline__ bool mbar_try(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  return done != 0;
}

// Bounded wait for an mbarrier phase. Gives up (false) when the CTA fail flag is set, or
// after timeout_ns of wall-clock time, in which case it sets the flag and reports the
// timeout for the grid.
// The fail flag and the clock are looked at once every 16 tries, so that a waiting warp
// issues few instructions (many warps wait at once and share the issue slots).
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, const StepSync& s,
                                          volatile int* fail) {
  if (mbar_try(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(mbar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*fail) return false;
      if (globaltimer_ns() - t0 > s.timeout_ns) {
        *fail = 1;
        give_up(s);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns, to every participating thread, the OR of x.
__device__ __forceinline__ bool named_bar_or(int id, int count, bool x) {
  uint32_t r;
  asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
               : "=r"(r) : "r"(static_cast<uint32_t>(x)), "r"(id), "r"(count) : "memory");
  return r != 0;
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

// 8 or 4 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                 "r"(v[7]) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4& w) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
               ::"r"(taddr), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w) : "memory");
}

// 32 consecutive columns from 8 raw 16-byte chunks (bf16 rows need no conversion).
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

// CH (4, 8 or 16) consecutive 32-bit columns of this thread's tensor-memory lane.
template <int CH>
__device__ __forceinline__ void tmem_ld(uint32_t a, float (&d)[CH]) {
  static_assert(CH == 4 || CH == 8 || CH == 16, "4, 8 or 16 columns");
  uint32_t r[CH];
  if constexpr (CH == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
  } else if constexpr (CH == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]) : "r"(a) : "memory");
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
                 "%10, %11, %12, %13, %14, %15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]) : "r"(a) : "memory");
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < CH; ++j) d[j] = __uint_as_float(r[j]);
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

// L2 policies: W2 rows are re-read at every position (keep them), base logits are read
// once (let them go first).
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ldg_keep(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u16_once(const uint16_t* ptr, uint64_t pol) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(ptr), "l"(pol));
  return v;
}

// Tensor-map copy of one box of the base logits [bs][K][V] (3-D) into shared memory,
// completion counted in bytes on `mbar`, with an L2 policy; executed by a whole warp,
// carried out by the leader lane (which also announces the bytes on `mbar`).
__device__ __forceinline__ void tma_load_3d_if(bool leader, void* dst, const CUtensorMap* map, int c0, int c1,
                                               int c2, uint64_t* mbar, uint32_t bytes, uint64_t pol) {
  asm volatile(
      "{ .reg .pred q; setp.ne.b32 q, %8, 0; "
      "@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%5], %7; "
      "@q cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6; }"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(mbar)), "l"(pol), "r"(bytes), "r"(static_cast<uint32_t>(leader))
      : "memory");
}

// L2 prefetch of one box of the base logits through the tensor map (leader lane).
__device__ __forceinline__ void tma_prefetch_3d_if(bool leader, const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("{ .reg .pred q; setp.ne.b32 q, %4, 0; "
               "@q cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}]; }"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
                 "r"(static_cast<uint32_t>(leader)) : "memory");
}

}  // namespace

// N = 16, 32 or 64 padded request rows (the MMA's N); each epilogue warp scores N / 4 of
// them. ROWS (with PROB): per-row modes or temperatures; the other instances score
// every column with the kernel's mode and temperature.
template <bool INT8, bool PROB, bool LOGITS, int N, bool ROWS>
__global__ void __launch_bounds__(kTcThreads, 1) walk_tc_kernel(const __grid_constant__ WalkParams p) {
  static_assert(PROB || !ROWS, "per-row settings come with sampled rows");
  constexpr int CPW = N / 4;                         // request columns per epilogue warp
  constexpr int kRowBytes = INT8 ? kRank : 2 * kRank;
  constexpr int kParts = kRowBytes / 128;            // 128-byte parts of a row (2 or 4)
  constexpr int kBlockBytes = 32 * kRowBytes;        // resident 32-row block
  constexpr uint32_t kIdesc = f16_idesc(INT8 ? 0u : 1u, N);

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start, by an offset from smem_raw so that every derived pointer
  // stays a shared-memory pointer
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int kDBufs = tc_dbufs(N);
  constexpr int NS = tc_base_stages(N);              // base-logit stages (tensor-map copies)
  constexpr int kStageBytes = kTile * N * 2;         // [N requests][128 rows] bf16
  unsigned char* b_s = smem;                                      // N x 512 bytes
  uint16_t* stage_s = reinterpret_cast<uint16_t*>(b_s + N * 512); // [NS][N][128] when base_tma
  unsigned char* w2s = b_s + N * 512 + (p.base_tma ? NS * kStageBytes : 0);  // resident blocks
  float* scale_s = reinterpret_cast<float*>(w2s + static_cast<size_t>(p.resident_rows) * kRowBytes);
  int* prev_s = reinterpret_cast<int*>(scale_s + (INT8 ? p.slice_cap : 0));   // [64]
  uint64_t* seed_s = reinterpret_cast<uint64_t*>(prev_s + 64);    // [64]
  uint64_t* best_s = seed_s + 64;                                 // [64]
  uint64_t* red_s = best_s + 64;                                  // [4][64]
  float2* inv_s = reinterpret_cast<float2*>(red_s + 4 * 64);       // 2^-s as two factors
  float* invT_s = reinterpret_cast<float*>(inv_s + 2);            // [64]
  uint64_t* gmask_s = reinterpret_cast<uint64_t*>(invT_s + 64);   // bit b: row b greedy
  uint64_t* mbar = gmask_s + 1;                                    // [24]
  uint64_t* a_full = mbar;        // [3], 4 producer-warp arrivals
  uint64_t* a_empty = mbar + 3;   // [3], 1 commit
  uint64_t* d_full = mbar + 6;    // [4], 1 commit
  uint64_t* d_empty = mbar + 10;  // [4], 16 epilogue-warp arrivals
  uint64_t* b_ready = mbar + 14;  // 1 arrival per position
  uint64_t* res_full = mbar + 15; // resident rows landed (bytes)
  uint64_t* s_full = mbar + 16;   // [4], 1 arrival + bytes
  uint64_t* s_empty = mbar + 20;  // [4], 16 epilogue-warp arrivals
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(mbar + 24);
  volatile int* fail = reinterpret_cast<volatile int*>(tbase_s + 1);
  int* flag = reinterpret_cast<int*>(tbase_s + 2);
  int* sh_amax = flag + 1;        // largest finite |e| of the batch, as fp32 bits

  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t v0 = slice_start(cta, G, p.V), v1 = slice_start(cta + 1, G, p.V);
  const int n = static_cast<int>(v1 - v0);
  const int nblk = (n + 31) / 32;
  const int res_blk = min(p.resident_rows / 32, nblk);
  const int str_blk = nblk - res_blk;                 // blocks 0 .. str_blk-1 are streamed
  const int T = (n + kTile - 1) / kTile;
  const unsigned char* w2g = (INT8 ? reinterpret_cast<const unsigned char*>(p.w2q)
                                   : reinterpret_cast<const unsigned char*>(p.w2)) +
                             static_cast<size_t>(v0) * kRowBytes;
  const bool skip0 = (p.sync.flags & DSPARK_FLAG_SKIP_ARRIVAL_CTA0) && cta == 0;

  // ---- set-up: zero B, scales, previous tokens, barriers, tensor memory
  for (int t = tid; t < N * 512 / 16; t += blockDim.x) reinterpret_cast<uint4*>(b_s)[t] = make_uint4(0, 0, 0, 0);
  if (INT8)
    for (int r = tid; r < n; r += blockDim.x) scale_s[r] = __ldg(p.scales + v0 + r);
  for (int t = tid; t < 64; t += blockDim.x) {
    const bool sampled = t < p.bs && row_sampled(p, PROB, t);
    seed_s[t] = sampled ? p.seeds[t] : 0ull;
    // 1/T rounded to fp32 from the double quotient, as the host does for the scalar T
    if constexpr (ROWS) invT_s[t] = sampled ? static_cast<float>(1.0 / static_cast<double>(row_temperature(p, t))) : 1.0f;
    if (t < p.bs) {
      const int32_t tok = p.prev[t];
      const bool okt = tok >= 0 && static_cast<int64_t>(tok) < p.V;
      const bool settings = row_settings_ok(p, PROB, t);
      prev_s[t] = okt && settings ? tok : -1;
      if (!okt && cta == 0) report(p.sync.status_dev, DSPARK_ERR_BAD_TOKEN);
      if (!settings && cta == 0) report(p.sync.status_dev, DSPARK_ERR_INVALID_ARG);
    }
  }
  if (tid == 0) {
    for (int b = 0; b < 24; ++b) {
      const uint32_t count = b < 3 ? 4u : (b >= 10 && b < 14) || b >= 20 ? 16u : 1u;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&mbar[b])), "r"(count));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *fail = 0;
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase_s;
  const bool res_tma = res_blk > 0;
  // Resident blocks: tensor-map copies of 32 rows x 128 bytes (128-byte swizzle), all
  // counted on res_full; the producers wait for them before the first resident block.
  if (tid == 0 && res_tma) {
    const uint32_t bytes = static_cast<uint32_t>(res_blk) * kBlockBytes;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(res_full)), "r"(bytes) : "memory");
    for (int rb = 0; rb < res_blk; ++rb) {
      const int row = static_cast<int>(v0) + 32 * (str_blk + rb);
#pragma unroll
      for (int h = 0; h < kParts; ++h)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(smem_u32(w2s + static_cast<size_t>(rb) * kBlockBytes + h * 4096)),
              "l"(reinterpret_cast<uint64_t>(&p.w2_map)), "r"(h * (INT8 ? 128 : 64)), "r"(row),
              "r"(smem_u32(res_full))
            : "memory");
    }
  }
  __syncwarp();  // warp 0 converges before its warp-collective work

  // Every role ends here once it has finished or given up: the resident copies land
  // (bounded), tensor memory is released, and a successful walk leaves the workspace
  // zeroed. Each role calls it from its own branch (the branches run with different
  // register limits).
  auto finish_cta = [&]() {
    if (warp == 0 && res_tma) {
      const uint64_t t0 = globaltimer_ns();
      while (!__all_sync(kFull, mbar_try(res_full, 0)) && !__any_sync(kFull, globaltimer_ns() - t0 >= p.sync.timeout_ns)) {}
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    if (!*fail) finish_walk(p.sync, p.K, p.bs, flag);
  };

  if (warp < kTcProducerWarps) {
    // ================================================================ producers
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcProducerRegs));
    const int q = warp;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const uint64_t keep = policy_evict_last();
    bool res_landed = !res_tma;
    int g = 0;  // global tile sequence number
    for (int i = 0; i < p.K && !__any_sync(kFull, *fail); ++i) {
      for (int t = 0; t < T; ++t, ++g) {
        const int abuf = g % kABufs;
        // (warp-uniform decisions: the tensor-memory stores below are warp-collective)
        if (g >= kABufs && __any_sync(kFull, !mbar_wait(&a_empty[abuf], ((g / kABufs) - 1) & 1, p.sync, fail))) break;
        tc_fence_after();
        const int blk = 4 * t + q;
        const int r = 32 * blk + lane;                  // row of this thread in the slice
        const uint32_t acol = tmem + lane_off + abuf * 128;
        if (blk < str_blk) {
          // streamed block: 8 chunks (128 bytes) of the row in flight at once, each
          // chunk stored as soon as it is converted
          const unsigned char* row = w2g + static_cast<size_t>(r) * kRowBytes;
#pragma unroll 1
          for (int hv = 0; hv < kParts; ++hv) {
            uint4 c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              c[j] = r < n ? ldg_keep(row + 128 * hv + 16 * j, keep) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if constexpr (INT8) {
                uint32_t v[8];
                int8x4_to_f16x4(c[j].x, v[0], v[1]);
                int8x4_to_f16x4(c[j].y, v[2], v[3]);
                int8x4_to_f16x4(c[j].z, v[4], v[5]);
                int8x4_to_f16x4(c[j].w, v[6], v[7]);
                tmem_st8(acol + 8 * (8 * hv + j), v);
              } else {
                tmem_st4(acol + 4 * (8 * hv + j), c[j]);
              }
            }
          }
        } else if (blk < nblk) {
          // resident block: shared memory, 128-byte swizzled parts
          if (!res_landed) {
            if (__any_sync(kFull, !mbar_wait(res_full, 0, p.sync, fail))) break;
            res_landed = true;
          }
          const int rr = r - 32 * str_blk;              // row within the resident area
          const unsigned char* rowb = w2s + static_cast<size_t>(rr >> 5) * kBlockBytes + (rr & 31) * 128;
          const int sw = rr & 7;
          // int8: the next pass's chunks are loaded while this pass converts
          [[maybe_unused]] uint4 cur[4];
          if constexpr (INT8) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              cur[j] = *reinterpret_cast<const uint4*>(rowb + ((j & 7) ^ sw) * 16);
          }
#pragma unroll
          for (int ps = 0; ps < 4; ++ps) {
            if constexpr (INT8) {
              uint4 nxt[4];
              if (ps < 3) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int c = (ps + 1) * 4 + j;     // logical 16-byte chunk of the row
                  nxt[j] = *reinterpret_cast<const uint4*>(rowb + (c >> 3) * 4096 + (((c & 7) ^ sw) << 4));
                }
              }
              uint32_t v[32];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                int8x4_to_f16x4(cur[j].x, v[8 * j + 0], v[8 * j + 1]);
                int8x4_to_f16x4(cur[j].y, v[8 * j + 2], v[8 * j + 3]);
                int8x4_to_f16x4(cur[j].z, v[8 * j + 4], v[8 * j + 5]);
                int8x4_to_f16x4(cur[j].w, v[8 * j + 6], v[8 * j + 7]);
              }
              tmem_st32(acol + 32 * ps, v);
              if (ps < 3) {
#pragma unroll
                for (int j = 0; j < 4; ++j) cur[j] = nxt[j];
              }
            } else {
              uint4 w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int c = ps * 8 + j;
                w[j] = *reinterpret_cast<const uint4*>(rowb + (c >> 3) * 4096 + (((c & 7) ^ sw) << 4));
              }
              tmem_st32_u4(acol + 32 * ps, w);
            }
          }
        } else {
          // past the slice: zero rows
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
#pragma unroll
          for (int ps = 0; ps < 4; ++ps) tmem_st32(acol + 32 * ps, v);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[abuf]);
      }
    }
    finish_cta();
  } else if (warp >= kIssuerWarp) {
    // ================================================================ MMA issue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTcIssuerRegs));
    // The whole warp runs each loop and waits (warp-uniform); one lane issues.
    const bool leader = lane == 0;
    if (warp == kIssuerWarp || warp == kIssuerWarp + 1) {
      // two issuing warps (on different SM sub-partitions) take alternate tiles
      const int parity = warp - kIssuerWarp;
      int g = 0;
      int last = -1;  // last tile whose MMAs were committed
      const uint32_t b_base = smem_u32(b_s);
      for (int i = 0; i < p.K && !__any_sync(kFull, *fail); ++i) {
        if (__any_sync(kFull, !mbar_wait(b_ready, i & 1, p.sync, fail))) break;
        bool ok = true;
        for (int t = 0; t < T; ++t, ++g) {
          if ((g & 1) != parity) continue;
          const int abuf = g % kABufs, dbuf = g % kDBufs;
          ok = !__any_sync(kFull, !mbar_wait(&a_full[abuf], (g / kABufs) & 1, p.sync, fail));
          if (ok && g >= kDBufs) ok = !__any_sync(kFull, !mbar_wait(&d_empty[dbuf], ((g / kDBufs) - 1) & 1, p.sync, fail));
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_col = tmem + abuf * 128;
          const uint32_t d_col = tmem + kColD + dbuf * N;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint64_t bd = sw128_desc(b_base + (kk / 4) * N * 128 + (kk % 4) * 32);
            mma_f16_if(leader, d_col, a_col + 8 * kk, bd, kIdesc, kk > 0 ? 1u : 0u);
          }
          mma_commit_if(leader, &d_full[dbuf]);
          mma_commit_if(leader, &a_empty[abuf]);
          last = g;
        }
        if (!ok) break;
      }
      // issued MMAs and their commits complete before tensor memory and the barriers
      // go (bounded wait)
      if (last >= 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!__all_sync(kFull, mbar_try(&a_empty[last % kABufs], (last / kABufs) & 1)) &&
               !__any_sync(kFull, globaltimer_ns() - t0 >= p.sync.timeout_ns)) {}
      }
    } else if (warp == kIssuerWarp + 2 && p.base_tma) {
      // ---------------------------------------------------- base-logit copies
      // Base logits do not depend on the tokens: this warp keeps the NS stages full,
      // running ahead of the epilogue across positions. Stage = the 128 rows of one
      // tile for all N request columns (columns past bs are filled with zeros).
      const uint64_t once = policy_evict_first();
      int k = 0;
      int issued = -1;
      for (int t = 0; t < T; ++t) tma_prefetch_3d_if(leader, &p.base_map, static_cast<int>(v0) + t * kTile, 0, 0);
      for (int i = 0; i < p.K && !__any_sync(kFull, *fail); ++i) {
        bool ok = true;
        // the next position's boxes towards L2 while this position's are copied
        if (i + 1 < p.K)
          for (int t = 0; t < T; ++t) tma_prefetch_3d_if(leader, &p.base_map, static_cast<int>(v0) + t * kTile, i + 1, 0);
        for (int t = 0; t < T; ++t, ++k) {
          const int sb = k % NS;
          if (k >= NS && !(ok = !__any_sync(kFull, !mbar_wait(&s_empty[sb], ((k / NS) - 1) & 1, p.sync, fail)))) break;
          tma_load_3d_if(leader, reinterpret_cast<unsigned char*>(stage_s) + sb * kStageBytes, &p.base_map,
                         static_cast<int>(v0) + t * kTile, i, 0, &s_full[sb], static_cast<uint32_t>(kStageBytes), once);
          issued = k;
        }
        if (!ok) break;
      }
      // copies in flight land before the CTA can leave (bounded)
      for (int k2 = max(0, issued - NS + 1); k2 <= issued; ++k2) {
        const uint64_t t0 = globaltimer_ns();
        while (!__all_sync(kFull, mbar_try(&s_full[k2 % NS], (k2 / NS) & 1)) &&
               !__any_sync(kFull, globaltimer_ns() - t0 >= p.sync.timeout_ns)) {}
      }
    }
    finish_cta();
  } else {
    // ================================================================ epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTcEpilogueRegs));
    const int ew = warp - kTcProducerWarps;   // 0..15
    const int etid = tid - kTcProducerWarps * 32;
    const int q = warp & 3;                   // tensor-memory lane quadrant
    const int cg = ew >> 2;                   // column group
    const int cb = cg * CPW;                  // first request column of the warp
    const int ncol = max(0, min(CPW, p.bs - cb));
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const uint64_t once = policy_evict_first();
    const size_t bstride = static_cast<size_t>(p.K) * static_cast<size_t>(p.V);
    int g = 0;

    // Embedding rows of the previous tokens -> B operand (K-major, 128-byte swizzle).
    // int8 W2: one power-of-two scale 2^s for the whole batch, with the largest finite
    // |e| of all rows in [2^14, 2^15) after scaling, converted to fp16.
    auto build_b = [&]() {
      uint4 wrow[4];
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int b = ew + kTcEpilogueWarps * r4;
        const int tok = b < p.bs ? prev_s[b] : -1;
        wrow[r4] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(tok) * kRank) + lane)
                            : make_uint4(0, 0, 0, 0);
      }
      int shift = 0;
      if constexpr (INT8) {
        float amax = 0.f;
#pragma unroll
        for (int r4 = 0; r4 < 4; ++r4) {
          const uint32_t ww[4] = {wrow[r4].x, wrow[r4].y, wrow[r4].z, wrow[r4].w};
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
        named_bar(kBarEpi, kEpiThreads);
        const float am = __int_as_float(*reinterpret_cast<volatile int*>(sh_amax));
        if (am > 0.f) {
          int ex;
          frexpf(am, &ex);  // am = f 2^ex, f in [0.5, 1)
          shift = 15 - ex;  // am 2^shift in [2^14, 2^15)
        }
      }
#pragma unroll
      for (int r4 = 0; r4 < 4; ++r4) {
        const int b = ew + kTcEpilogueWarps * r4;
        if (b >= p.bs) break;
        uint4 w = wrow[r4];
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
      if (etid == 0)
        *inv_s = make_float2(__int_as_float(((-shift) / 2 + 127) << 23),
                             __int_as_float(((-shift) - (-shift) / 2 + 127) << 23));
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_bar(kBarEpi, kEpiThreads);  // B written and visible to the tensor core; 2^-s published
      if (etid == 0) {
        *sh_amax = 0;
        mbar_arrive(b_ready);
      }
    };

    // Base logits of the first two positions towards L2; later ones two positions ahead.
    auto prefetch_base = [&](int i) {
      if (i >= p.K || n <= 0) return;
      const int lines = (n * 2 + 127) / 128 + 1;  // 128-byte lines of one row's slice
      for (int b = ew; b < p.bs; b += kTcEpilogueWarps) {
        const uint16_t* row = p.base + (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v0;
        for (int l = lane; l < lines; l += 32) prefetch_l2(row + min(64 * l, n - 1));
      }
    };
    if (!p.base_tma) {  // (with base_tma the copying thread prefetches whole boxes)
      prefetch_base(0);
      prefetch_base(1);
    }
    build_b();

    bool walked = true;  // every position of this CTA completed
    for (int i = 0; i < p.K; ++i) {
      if (i + 2 < p.K && !p.base_tma) prefetch_base(i + 2);
      const uint16_t* brow = p.base + static_cast<size_t>(i) * p.V + v0;  // + b K V + row
      [[maybe_unused]] const uint32_t wg = ROWS ? static_cast<uint32_t>(*gmask_s >> cb) : 0u;  // greedy columns
      const float2 inv = inv_s[0];
      float bv[CPW];
      uint32_t bt[(CPW + 3) / 4];
#pragma unroll
      for (int j = 0; j < CPW; ++j) bv[j] = -INFINITY;
#pragma unroll
      for (int w = 0; w < (CPW + 3) / 4; ++w) bt[w] = 0u;
      // base logits of this thread's row in the warp's columns, loaded one tile ahead
      uint32_t bnext[CPW];
      auto load_base = [&](int t) {
        const int r = t * kTile + 32 * q + lane;
        const bool valid = r < n;
#pragma unroll
        for (int j = 0; j < CPW; ++j)
          bnext[j] = (valid && j < ncol) ? ldg_u16_once(brow + static_cast<size_t>(cb + j) * bstride + r, once) : 0u;
      };
      if (T > 0 && !p.base_tma) load_base(0);
      bool ok = !__any_sync(kFull, *fail);  // warp-uniform: the tile loop is warp-collective
      float d[CPW];        // the contraction D of this thread's row, the warp's columns
      uint32_t braw[CPW];  // base logits (bf16 bits) of this thread's row, the warp's columns
      // Scores of columns 4 h4 .. 4 h4 + 3 of tile t and the running-maximum update.
      // MASK: the tile reaches past the slice, rows past it score -inf. Columns past bs
      // are scored too and never stored.
      auto score_group = [&](auto mask_tag, int t, int h4, float c, bool valid, uint32_t trep) {
        constexpr bool MASK = decltype(mask_tag)::value;
        [[maybe_unused]] const int r = t * kTile + 32 * q + lane;  // (the logit store's row)
        float sc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 4 * h4 + k;
          const float bvl = __uint_as_float(braw[j] << 16);
          float l;
          if constexpr (INT8) l = __fmaf_rn(d[j], c, bvl);
          else l = __fadd_rn(d[j], bvl);
          if constexpr (MASK) l = valid ? l : -INFINITY;
          [[maybe_unused]] const uint16_t lh = f32_to_bf16_bits(l);
          if constexpr (LOGITS) {
            if (valid && j < ncol)
              p.logits[static_cast<size_t>(cb + j) * bstride + static_cast<size_t>(i) * p.V + v0 + r] = lh;
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
          // Gumbel noise: lane 4m + k draws the Philox block of rows 4m..4m+3 (of the
          // warp's 32) and column 4 h4 + k, then a 4 x 4 transpose inside the lane quad
          // leaves every lane the draws of its own row for these 4 columns.
          const uint32_t m = (static_cast<uint32_t>(v0) + t * kTile + 32 * q) / 4 + (lane >> 2);
          const int bq = cb + 4 * h4 + (lane & 3);
          const uint4 w = philox_block(seed_s[bq], bq, i, m);
          float g4[4] = {gumbel_from_word(w.x), gumbel_from_word(w.y), gumbel_from_word(w.z),
                         gumbel_from_word(w.w)};
          transpose4(g4, lane);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (!ROWS || !((wg >> (4 * h4 + k)) & 1u)) sc[k] = __fadd_rn(sc[k], g4[k]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 4 * h4 + k;
          float nv;
          asm("max.NaN.f32 %0, %1, %2;" : "=f"(nv) : "f"(bv[j]), "f"(sc[k]));
          // the tile is rewritten when the maximum changes (an unordered compare, so the
          // first NaN counts) unless it already is NaN; equal values never rewrite it,
          // so the first maximum (smallest tile) stays
          asm("{ .reg .pred r, u; setp.num.f32 r, %1, %1; setp.neu.and.f32 u, %2, %1, r; "
              "@u lop3.b32 %0, %0, %3, %4, 0xB8; }"
              : "+r"(bt[j >> 2]) : "f"(bv[j]), "f"(nv), "r"(0xFFu << (8 * (j & 3))), "r"(trep));
          bv[j] = nv;
        }
      };
      for (int t = 0; t < T && ok; ++t, ++g) {
        const int dbuf = g % kDBufs;
        const int sb = g % NS;
        if (p.base_tma) {
          // this tile's base logits from the stage ring
          if (__any_sync(kFull, !mbar_wait(&s_full[sb], (g / NS) & 1, p.sync, fail))) { ok = false; break; }
          const uint16_t* st = stage_s + static_cast<size_t>(sb) * (kStageBytes / 2) + cb * kTile + 32 * q + lane;
#pragma unroll
          for (int j = 0; j < CPW; ++j) braw[j] = st[j * kTile];
        } else {
#pragma unroll
          for (int j = 0; j < CPW; ++j) braw[j] = bnext[j];
          if (t + 1 < T) load_base(t + 1);
        }
        if (__any_sync(kFull, !mbar_wait(&d_full[dbuf], (g / kDBufs) & 1, p.sync, fail))) { ok = false; break; }
        tc_fence_after();
        tmem_ld<CPW>(tmem + lane_off + kColD + dbuf * N + cb, d);
        // D and the base logits are in registers: both buffers go back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&d_empty[dbuf]);
          if (p.base_tma) mbar_arrive(&s_empty[sb]);
        }
        const int r = t * kTile + 32 * q + lane;
        const bool valid = r < n;
        [[maybe_unused]] float c = 1.f;
        if constexpr (INT8) c = __fmul_rn(__fmul_rn(valid ? scale_s[r] : 0.f, inv.x), inv.y);
        const uint32_t trep = static_cast<uint32_t>(t) * 0x01010101u;
        if ((t + 1) * kTile <= n) {
#pragma unroll
          for (int h4 = 0; h4 < CPW / 4; ++h4) score_group(std::false_type{}, t, h4, c, valid, trep);
        } else {
#pragma unroll
          for (int h4 = 0; h4 < CPW / 4; ++h4) score_group(std::true_type{}, t, h4, c, valid, trep);
        }
      }
      // -------- per column: (orderable key, first index) maximum over the warp's rows;
      // the first index among the lanes that reach it is the smallest (tile, lane)
      if (ok) {
        // independent chains per column (no early exit, so they interleave); columns
        // past bs are reduced too and not stored
        uint32_t key[CPW], pos[CPW];
#pragma unroll
        for (int j = 0; j < CPW; ++j) key[j] = order_key(bv[j]);
#pragma unroll
        for (int j = 0; j < CPW; ++j) {
          const uint32_t kmax = __reduce_max_sync(kFull, key[j]);
          const uint32_t tj = (bt[j >> 2] >> (8 * (j & 3))) & 0xFFu;
          pos[j] = key[j] == kmax ? ((tj << 5) | static_cast<uint32_t>(lane)) : 0xFFFFFFFFu;
          key[j] = kmax;
        }
#pragma unroll
        for (int j = 0; j < CPW; ++j) pos[j] = __reduce_min_sync(kFull, pos[j]);
        if (lane == 0) {
#pragma unroll
          for (int j = 0; j < CPW; ++j)
            if (j < ncol)
              red_s[q * 64 + cb + j] =
                  pack_best(key[j], static_cast<uint32_t>(v0) + 32u * q + (pos[j] & 31u) + (pos[j] >> 5) * kTile);
        }
      }
      if (named_bar_or(kBarEpi, kEpiThreads, !ok || *fail)) { walked = false; break; }
      // -------- grid exchange of the per-row words: one atomicMax per (CTA, row), then
      // the bounded step barrier
      uint64_t* slots_i = p.sync.slots + static_cast<size_t>(i) * p.bs;
      if (etid < p.bs) {
        uint64_t x = umax64(umax64(red_s[etid], red_s[64 + etid]), umax64(red_s[128 + etid], red_s[192 + etid]));
        if (prev_s[etid] < 0 || n <= 0) x = 0ull;  // dead row, or a CTA without vocabulary rows
        if (x != 0ull) {
          atomicMax(reinterpret_cast<unsigned long long*>(slots_i + etid), static_cast<unsigned long long>(x));
          if (i + 1 < p.K) {  // the grid's winner is one of the local winners: its W1 row towards L2
            const uint16_t* w1row = p.w1 + static_cast<size_t>(unpack_idx(x)) * kRank;
#pragma unroll
            for (int l4 = 0; l4 < 4; ++l4) prefetch_l2(w1row + 64 * l4);
          }
        }
      }
      named_bar(kBarEpi, kEpiThreads);
      if (ew == 0) {
        // the whole warp waits (lane 0 polls, the value is broadcast): no lane waits
        // at a barrier for another lane of its warp
        uint32_t* ctr = p.sync.counter(i);
        // the release add is cumulative: the named barrier above orders every thread's
        // atomicMax before it
        if (lane == 0 && !(skip0 && i == 0)) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        __syncwarp();
        bool good = true;
        uint64_t t0 = 0;
        for (uint32_t it = 0;; ++it) {
          uint32_t c = 0;
          if (lane == 0) c = ld_acquire_u32(ctr);
          if (__shfl_sync(kFull, c, 0) >= p.sync.grid) break;
          if ((it & 63u) != 63u) continue;
          uint32_t stop = 0;
          if (lane == 0) {
            if (t0 == 0) t0 = globaltimer_ns();
            if (*reinterpret_cast<volatile uint32_t*>(&p.sync.hdr->abort) != 0u || *fail) stop = 1;
            else if (globaltimer_ns() - t0 > p.sync.timeout_ns) { give_up(p.sync); stop = 1; }
          }
          if (__shfl_sync(kFull, stop, 0)) { good = false; break; }
        }
        if (lane == 0) {
          if (!good) *fail = 1;
          *flag = good ? 1 : 0;
        }
      }
      named_bar(kBarEpi, kEpiThreads);
      if (*flag == 0) { walked = false; break; }
      if (etid < p.bs) {
        const int tok = prev_s[etid] >= 0 ? unpack_idx(ld_relaxed_u64(slots_i + etid)) : -1;
        prev_s[etid] = tok;
        if (cta == 0) p.tokens[static_cast<size_t>(etid) * p.K + i] = tok;
        // reset-behind: every CTA has passed step i's barrier, so nobody reads step
        // i-1's slots or counter again
        if (cta == 0 && i >= 1) p.sync.slots[static_cast<size_t>(i - 1) * p.bs + etid] = 0ull;
      }
      if (cta == 0 && i >= 1 && etid == 0) *p.sync.counter(i - 1) = 0u;
      named_bar(kBarEpi, kEpiThreads);  // new prev tokens visible
      if (i + 1 < p.K) build_b();
    }
    if (!walked) *fail = 1;
    finish_cta();
  }
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
