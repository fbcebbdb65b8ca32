// The drafter's LM head fused with the top-k candidate selection (vLLM PR #49969,
// "Purpose": the base logits of every draft position come from a dense LM-head GEMM,
// and the top-k candidates are selected from them once). Instead of writing the dense
// [M, V] logits and reading them back, the selection happens in the GEMM's epilogue:
//
//   1. sample pass: the same GEMM over every kSampleStride-th LM-head row; the logits
//      of those S rows are stored ([M, S] fp32, small);
//   2. pivot: per hidden row m, the j-th largest sampled key, with j chosen so that far
//      more than k of the V logits lie at or above it (keys: order-preserving uint32 of
//      the fp32 logit, NaN largest, -0 equal to +0);
//   3. filter pass: the GEMM over all V rows; the epilogue appends every logit whose key
//      reaches the row's pivot to the row's list, as the packed word {key, 2^32-1-v}
//      (the largest words are the top-k in the method's order: larger value first,
//      smaller index among equal values);
//   4. select: per row, the k largest packed words of the list by radix selection ->
//      the candidates and their fp32 logits. A row whose list holds fewer than k words
//      or overflowed takes the exact path: its logits recomputed on CUDA cores for a
//      radix selection over the whole row and an index-ordered pass for the ties.
//
// The GEMM: D[128 LM-head rows x up to 512 hidden rows] = A . B^T with A = 128 rows of
// the LM head (bf16, K-major, 128-byte swizzle, staged by tensor-map copies) and B = the
// hidden rows (two N parts of up to 256), accumulated in fp32 in tensor memory over
// 64-wide chunks of d (tcgen05 kind::f16, bf16 inputs). Warp 0 copies, warp 1 issues
// the MMAs, warps 2-5 run the epilogue; two stages of A and B.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "lmhead.cuh"

namespace dspark {

namespace {

constexpr int kLmTile = 128;          // LM-head rows per tile (the MMA's M)
constexpr int kLmChunk = 64;          // d elements per stage (128 bytes of bf16)
constexpr int kLmStages = 2;
constexpr int kLmBStageBytes = 2 * 256 * 128;   // two N parts of 256 hidden rows
constexpr int kLmAStageBytes = kLmTile * 128;
constexpr uint32_t kLmTmemCols = 512;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, M = 128.
__host__ __device__ constexpr uint32_t bf16_idesc(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(kLmTile >> 4) << 24);
}
__device__ __forceinline__ bool mbar_try(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  return done != 0;
}
// Bounded wait; on timeout sets the CTA fail flag and reports DSPARK_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, const LmParams& p, volatile int* fail) {
  if (mbar_try(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(mbar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*fail) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        *fail = 1;
        report(p.status_dev, DSPARK_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(mbar)) : "memory");
}

// Inverse of order_key (the key of -0 is the key of +0: it returns +0).
__device__ __forceinline__ float key_value(uint32_t key) {
  if (key == 0xFFFFFFFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

}  // namespace

// MODE 0: sample pass (rows r * stride of the LM head, logits stored); MODE 1: filter
// pass (every row, logits at or above the row's pivot appended to its list).
template <int MODE>
__global__ void __launch_bounds__(192, 1) lmhead_gemm_kernel(const __grid_constant__ LmParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* a_s = smem;                                         // [stages][128 x 128 B]
  unsigned char* b_s = smem + kLmStages * kLmAStageBytes;            // [stages][2 x 256 x 128 B]
  uint32_t* piv_s = reinterpret_cast<uint32_t*>(b_s + kLmStages * kLmBStageBytes);  // [4 warps][512]
  uint64_t* mbar = reinterpret_cast<uint64_t*>(piv_s + 4 * 512);
  uint64_t* full = mbar;           // [stages] 1 arrival + bytes
  uint64_t* empty = mbar + 2;      // [stages] 1 commit
  uint64_t* dfull = mbar + 4;      // 1 commit
  uint64_t* dempty = mbar + 5;     // 4 epilogue-warp arrivals
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(mbar + 6);
  volatile int* fail = reinterpret_cast<volatile int*>(tbase_s + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rows = MODE == 0 ? p.S : p.V;                       // LM-head rows of this pass
  const int tiles = static_cast<int>((rows + kLmTile - 1) / kLmTile);
  const int mchunks = (p.M + 511) / 512;
  const int units = tiles * mchunks;
  const int nk = p.d / kLmChunk;

  if (tid == 0) {
    for (int b = 0; b < 6; ++b)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&mbar[b])), "r"(b == 5 ? 4u : 1u));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *fail = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tbase_s)), "r"(kLmTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tbase_s;
  const CUtensorMap* amap = MODE == 0 ? &p.ws_map : &p.w_map;

  if (warp == 0) {
    // ------------------------------------------------------------ tensor-map copies
    const bool leader = lane == 0;
    int g = 0;  // global chunk counter
    for (int u = blockIdx.x; u < units && !__any_sync(kFull, *fail); u += gridDim.x) {
      const int tile = u / mchunks, mc = u % mchunks;
      const int m0 = mc * 512;
      const int nparts = p.M - m0 > 256 ? 2 : 1;
      const uint32_t bytes = kLmAStageBytes + nparts * 256 * 128;
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc, ++g) {
        const int s = g % kLmStages;
        if (g >= kLmStages && (ok = !__any_sync(kFull, !mbar_wait(&empty[s], ((g / kLmStages) - 1) & 1, p, fail))) == false) break;
        asm volatile(
            "{ .reg .pred q; setp.ne.b32 q, %2, 0; @q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1; }"
            ::"r"(smem_u32(&full[s])), "r"(bytes), "r"(static_cast<uint32_t>(leader)) : "memory");
        asm volatile(
            "{ .reg .pred q; setp.ne.b32 q, %5, 0; "
            "@q cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4]; }"
            ::"r"(smem_u32(a_s + s * kLmAStageBytes)), "l"(reinterpret_cast<uint64_t>(amap)),
              "r"(kc * kLmChunk), "r"(tile * kLmTile), "r"(smem_u32(&full[s])), "r"(static_cast<uint32_t>(leader))
            : "memory");
        for (int part = 0; part < nparts; ++part)
          asm volatile(
              "{ .reg .pred q; setp.ne.b32 q, %5, 0; "
              "@q cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4]; }"
              ::"r"(smem_u32(b_s + s * kLmBStageBytes + part * 256 * 128)), "l"(reinterpret_cast<uint64_t>(&p.h_map)),
                "r"(kc * kLmChunk), "r"(m0 + 256 * part), "r"(smem_u32(&full[s])), "r"(static_cast<uint32_t>(leader))
              : "memory");
      }
      if (!ok) break;
    }
    // copies still in flight land before the CTA leaves (bounded)
    for (int s = 0; s < kLmStages; ++s) {
      if (g - 1 - s < 0) continue;
      const int gl = g - 1 - s;
      const uint64_t t0 = globaltimer_ns();
      while (!__all_sync(kFull, mbar_try(&full[gl % kLmStages], (gl / kLmStages) & 1)) &&
             !__any_sync(kFull, globaltimer_ns() - t0 >= p.timeout_ns)) {}
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    const bool leader = lane == 0;
    int g = 0, un = 0, last = -1;
    for (int u = blockIdx.x; u < units && !__any_sync(kFull, *fail); u += gridDim.x, ++un) {
      const int mc = u % mchunks;
      const int m0 = mc * 512;
      const int mrows = min(512, p.M - m0);
      const int n0 = (min(256, mrows) + 15) & ~15;
      const int n1 = mrows > 256 ? ((mrows - 256 + 15) & ~15) : 0;
      if (un >= 1 && __any_sync(kFull, !mbar_wait(dempty, (un - 1) & 1, p, fail))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc, ++g) {
        const int s = g % kLmStages;
        if (__any_sync(kFull, !mbar_wait(&full[s], (g / kLmStages) & 1, p, fail))) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a0 = smem_u32(a_s + s * kLmAStageBytes), b0 = smem_u32(b_s + s * kLmBStageBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sw128_desc(a0 + kk * 32);
          const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
          for (int part = 0; part < 2; ++part) {
            const int np = part == 0 ? n0 : n1;
            if (np == 0) continue;
            const uint64_t bd = sw128_desc(b0 + part * 256 * 128 + kk * 32);
            asm volatile(
                "{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0; "
                "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                ::"r"(tmem + part * 256), "l"(ad), "l"(bd), "r"(bf16_idesc(np)), "r"(acc),
                  "r"(static_cast<uint32_t>(leader)) : "memory");
          }
        }
        asm volatile("{ .reg .pred q; setp.ne.b32 q, %1, 0; "
                     "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
                     ::"r"(smem_u32(&empty[s])), "r"(static_cast<uint32_t>(leader)) : "memory");
      }
      if (!ok) break;
      asm volatile("{ .reg .pred q; setp.ne.b32 q, %1, 0; "
                   "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }"
                   ::"r"(smem_u32(dfull)), "r"(static_cast<uint32_t>(leader)) : "memory");
      last = un;
    }
    if (last >= 0) {  // the last unit's MMAs complete before tensor memory goes (bounded)
      const uint64_t t0 = globaltimer_ns();
      while (!__all_sync(kFull, mbar_try(dfull, last & 1)) && !__any_sync(kFull, globaltimer_ns() - t0 >= p.timeout_ns)) {}
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // tensor-memory lane quadrant (warps 2..5 -> 2, 3, 0, 1)
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    uint32_t* piv_w = piv_s + 512 * (warp - 2);  // this warp's copy of the chunk's pivots
    int un = 0;
    for (int u = blockIdx.x; u < units && !__any_sync(kFull, *fail); u += gridDim.x, ++un) {
      const int tile = u / mchunks, mc = u % mchunks;
      const int m0 = mc * 512;
      const int mrows = min(512, p.M - m0);
      if (MODE == 1) {
        __syncwarp();  // the previous unit's pivots are read
        for (int t = lane; t < mrows; t += 32) piv_w[t] = p.pivot[m0 + t];
        __syncwarp();
      }
      if (__any_sync(kFull, !mbar_wait(dfull, un & 1, p, fail))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int64_t r = static_cast<int64_t>(tile) * kLmTile + 32 * q + lane;  // LM-head row of the pass
      const bool rvalid = r < rows;
      for (int c0 = 0; c0 < mrows; c0 += 32) {
        const uint32_t col = c0;  // hidden row 256 + j of part 1 sits in column 256 + j
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
            "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
              "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
            : "r"(tmem + lane_off + col) : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int m = c0 + j;  // hidden row within the chunk
          if (m >= mrows || !rvalid) continue;
          const float x = __uint_as_float(v[j]);
          if constexpr (MODE == 0) {
            p.sample[static_cast<size_t>(m0 + m) * p.S + r] = x;
          } else {
            const uint32_t key = order_key(x);
            if (key >= piv_w[m]) {
              const uint32_t pos = atomicAdd(p.cnt + m0 + m, 1u);
              if (pos < static_cast<uint32_t>(p.cap))
                p.list[static_cast<size_t>(m0 + m) * p.cap + pos] = pack_best(key, static_cast<uint32_t>(r));
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kLmTmemCols) : "memory");
}

namespace {

constexpr int kSelThreads = 512;

// Block-wide radix selection step: given a 256-bin histogram in shared memory and the
// number of items strictly above the current prefix range, the bin holding the
// `rank`-th largest item (1-based) and the count of items above that bin.
__device__ __forceinline__ void pick_bin(const int* hist, int above, int rank, int* out_bin, int* out_above) {
  int acc = above, bin = 0;
  for (int h = 255; h >= 0; --h) {
    if (acc + hist[h] >= rank) { bin = h; break; }
    acc += hist[h];
  }
  *out_bin = bin;
  *out_above = acc;
}

// fp32 dot product of hidden row m and LM-head row v on CUDA cores (fixed order).
__device__ __forceinline__ float dot_row(const LmParams& p, int m, int64_t v) {
  const uint4* h = reinterpret_cast<const uint4*>(p.hidden + static_cast<size_t>(m) * p.d);
  const uint4* w = reinterpret_cast<const uint4*>(p.lm_head + static_cast<size_t>(v) * p.d);
  float acc = 0.f;
  for (int c = 0; c < p.d / 8; ++c) {
    const uint4 a = __ldg(h + c), b = __ldg(w + c);
    const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc = __fmaf_rn(bf16_lo(aa[t]), bf16_lo(bb[t]), acc);
      acc = __fmaf_rn(bf16_hi(aa[t]), bf16_hi(bb[t]), acc);
    }
  }
  return acc;
}

}  // namespace

// Per hidden row: the pivot key = the j-th largest key of the row's sampled logits (one
// CTA per row, radix selection over four bytes), and the row's list counter zeroed.
__global__ void __launch_bounds__(kSelThreads) lmhead_pivot_kernel(const LmParams p, int j) {
  __shared__ int hist[256];
  __shared__ int sel[2];
  const int m = blockIdx.x;
  const float* x = p.sample + static_cast<size_t>(m) * p.S;
  uint32_t prefix = 0;
  int above = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int sh = 24 - 8 * pass;
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < p.S; s += blockDim.x) {
      const uint32_t key = order_key(x[s]);
      if (pass == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&hist[(key >> sh) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) pick_bin(hist, above, j, &sel[0], &sel[1]);
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(sel[0]);
    above = sel[1];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.pivot[m] = prefix;
    p.cnt[m] = 0u;
  }
}

// Per hidden row: the k largest packed words of its list (one CTA per row, the list in
// shared memory, radix selection over eight bytes), or the exact path over the whole
// row when the list is short, overflowed or the fallback is forced.
__global__ void __launch_bounds__(kSelThreads) lmhead_select_kernel(const LmParams p) {
  extern __shared__ __align__(1024) unsigned char sel_raw[];
  uint64_t* words = reinterpret_cast<uint64_t*>(sel_raw);             // [cap]
  __shared__ int hist[256];
  __shared__ int sel[2];
  __shared__ int outpos;
  const int m = blockIdx.x;
  const int k = p.k;
  const uint32_t n_all = p.cnt[m];
  const bool exact = (p.flags & kLmForceExact) || n_all < static_cast<uint32_t>(k) ||
                     n_all > static_cast<uint32_t>(p.cap);
  int32_t* cand = p.cand + static_cast<size_t>(m) * k;
  float* cbase = p.cand_base + static_cast<size_t>(m) * k;
  if (threadIdx.x == 0) outpos = 0;
  if (!exact) {
    const int n = static_cast<int>(n_all);
    for (int t = threadIdx.x; t < n; t += blockDim.x) words[t] = p.list[static_cast<size_t>(m) * p.cap + t];
    __syncthreads();
    uint64_t prefix = 0;
    int above = 0;
    for (int pass = 0; pass < 8; ++pass) {
      const int sh = 56 - 8 * pass;
      for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
      __syncthreads();
      for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const uint64_t w = words[t];
        if (pass == 0 || (w >> (sh + 8)) == prefix) atomicAdd(&hist[(w >> sh) & 0xFFu], 1);
      }
      __syncthreads();
      if (threadIdx.x == 0) pick_bin(hist, above, k, &sel[0], &sel[1]);
      __syncthreads();
      prefix = (prefix << 8) | static_cast<uint64_t>(sel[0]);
      above = sel[1];
      __syncthreads();
    }
    // words are distinct (one per vocabulary entry): exactly k are >= the k-th largest
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
      const uint64_t w = words[t];
      if (w >= prefix) {
        const int pos = atomicAdd(&outpos, 1);
        cand[pos] = unpack_idx(w);
        cbase[pos] = key_value(static_cast<uint32_t>(w >> 32));
      }
    }
    return;
  }
  if (threadIdx.x == 0 && p.stats) atomicAdd(p.stats + (n_all > static_cast<uint32_t>(p.cap) ? 1 : 0), 1);
  // exact path: radix selection of the k-th largest key over the whole recomputed row,
  // then an index-ordered pass taking keys above it and the first ties
  uint32_t prefix = 0;
  int above = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int sh = 24 - 8 * pass;
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    __syncthreads();
    for (int64_t v = threadIdx.x; v < p.V; v += blockDim.x) {
      const uint32_t key = order_key(dot_row(p, m, v));
      if (pass == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&hist[(key >> sh) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) pick_bin(hist, above, k, &sel[0], &sel[1]);
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(sel[0]);
    above = sel[1];
    __syncthreads();
  }
  const uint32_t thr = prefix;
  const int need_eq = k - above;  // entries equal to thr still to take (>= 1)
  __shared__ int eq_seen;
  if (threadIdx.x == 0) eq_seen = 0;
  __syncthreads();
  for (int64_t v0 = 0; v0 < p.V; v0 += blockDim.x) {
    const int64_t v = v0 + threadIdx.x;
    const float x = v < p.V ? dot_row(p, m, v) : 0.f;
    const uint32_t key = v < p.V ? order_key(x) : 0u;
    const bool eq = v < p.V && key == thr;
    // ties in index order: rank among this chunk's equal keys by a block scan
    const uint32_t ball = __ballot_sync(kFull, eq);
    __shared__ int warp_eq[kSelThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) warp_eq[warp] = __popc(ball);
    __syncthreads();
    int before = eq_seen;
    for (int w = 0; w < warp; ++w) before += warp_eq[w];
    before += __popc(ball & ((1u << lane) - 1u));
    const bool take = (v < p.V) && (key > thr || (eq && before < need_eq));
    if (take) {
      const int pos = atomicAdd(&outpos, 1);
      cand[pos] = static_cast<int32_t>(v);
      cbase[pos] = x;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < kSelThreads / 32; ++w) tot += warp_eq[w];
      eq_seen += tot;
    }
    __syncthreads();
  }
}

size_t lmhead_select_smem(int cap) { return static_cast<size_t>(cap) * 8; }

cudaError_t launch_lmhead(LmParams& p, int sms, int pivot_rank, cudaStream_t stream) {
  const size_t smem = 1024 + kLmStages * (kLmAStageBytes + kLmBStageBytes) + 4 * 512 * 4 + 6 * 8 + 16;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(lmhead_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(lmhead_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) != cudaSuccess)
    return e;
  const size_t ssmem = lmhead_select_smem(p.cap);
  if ((e = cudaFuncSetAttribute(lmhead_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(ssmem))) != cudaSuccess)
    return e;
  const int mchunks = (p.M + 511) / 512;
  const int units0 = static_cast<int>((p.S + kLmTile - 1) / kLmTile) * mchunks;
  const int units1 = static_cast<int>((p.V + kLmTile - 1) / kLmTile) * mchunks;
  lmhead_gemm_kernel<0><<<min(sms, units0), 192, smem, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  lmhead_pivot_kernel<<<p.M, kSelThreads, 0, stream>>>(p, pivot_rank);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  lmhead_gemm_kernel<1><<<min(sms, units1), 192, smem, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  lmhead_select_kernel<<<p.M, kSelThreads, ssmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dspark

namespace dspark {

// draft_logits rows of the fused top-k path start as -inf (the walk writes the
// candidates' values).
__global__ void fill_neg_inf_kernel(uint16_t* x, size_t n) {
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<size_t>(gridDim.x) * blockDim.x)
    x[t] = 0xFF80u;
}

cudaError_t launch_fill_neg_inf(uint16_t* x, size_t n, cudaStream_t stream) {
  const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
  fill_neg_inf_kernel<<<blocks, 256, 0, stream>>>(x, n);
  return cudaGetLastError();
}

}  // namespace dspark
