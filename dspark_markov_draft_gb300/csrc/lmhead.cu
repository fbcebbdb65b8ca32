// The drafter's LM head fused with the top-k candidate selection (vLLM PR #49969,
// "Purpose": the base logits of every draft position come from a dense LM-head GEMM,
// and the top-k candidates are selected from them once). Instead of writing the dense
// [M, V] logits and reading them back, the selection happens in the GEMM's epilogue:
//
//   1. sample pass: the same GEMM over every kSampleStride-th LM-head row; the logits
//      of those S rows are stored ([M, S] fp32, small);
//   2. pivot: per hidden row m, a key with at least j sampled keys at or above it (the
//      j-th largest, resolved to its top bits), j chosen so that more than k of the V
//      logits lie at or above it (keys: order-preserving uint32 of the fp32 logit, NaN
//      largest, -0 equal to +0);
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
// 64-wide chunks of d (tcgen05 kind::f16, bf16 inputs). Warp 0 copies (and prefetches
// the LM-head chunks a few stages ahead into L2), warp 1 issues the MMAs, sixteen warps
// read the accumulator back; as many stages as shared memory holds (three at 448 hidden
// rows). The epilogue is short next to a tile's MMAs: each of its warps reads 32 x 32
// accumulators per step and tests them against per-column pivots broadcast by shuffles.
//
// Passes 2-4 are launched as programmatic dependents of the pass before them: a pass may
// be scheduled once every CTA of the previous one has started (or, after the filter
// pass, finished its tiles), so its launch and set-up overlap the previous pass's end,
// and it waits for the previous pass to complete (griddepcontrol.wait) before reading
// what that pass wrote. In the filter pass only the epilogue waits (it reads the pivots
// and appends to the lists the pivot pass reset): the copies and MMAs of its first
// tiles read only the inputs, which the sample pass -- launched in stream order --
// already found complete.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "lmhead.cuh"

namespace dspark {

namespace {

constexpr int kLmTile = 128;          // LM-head rows per tile (the MMA's M)
constexpr int kLmChunk = 64;          // d elements per stage (128 bytes of bf16)
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
// Programmatic dependent launch: let the next pass be scheduled before this one
// completes (it waits for this pass with wait_previous_kernel before reading its output).
__device__ __forceinline__ void allow_next_pass() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t bf16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// CLUSTER: acquire at cluster scope (arrivals that come from the other CTA of the pair).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try(uint64_t* mbar, uint32_t parity) {
  uint32_t done;
  if (CLUSTER)
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  else
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
  return done != 0;
}
// Bounded wait; on timeout sets the CTA fail flag and reports DSPARK_ERR_TIMEOUT.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, const LmParams& p, volatile int* fail) {
  if (mbar_try<CLUSTER>(mbar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try<CLUSTER>(mbar, parity)) return true;
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
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Every thread of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of `p`'s counterpart in the pair's CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Tensor-map copy of one 2-D box into this CTA's shared memory, its bytes counted on a
// barrier of either CTA of the pair (`bar`: shared::cluster address); leader lane only.
__device__ __forceinline__ void tma_2d_pair_if(uint32_t leader, void* dst, const CUtensorMap* map, int x, int y,
                                               uint32_t bar) {
  asm volatile(
      "{ .reg .pred q; setp.ne.b32 q, %5, 0; "
      "@q cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
      "[%0], [%1, {%2, %3}], [%4]; }"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_2d_if(uint32_t leader, const CUtensorMap* map, int x, int y) {
  asm volatile("{ .reg .pred q; setp.ne.b32 q, %3, 0; @q cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}]; }"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(leader) : "memory");
}
// Arrive on `bar` in both CTAs of the pair once the paired MMAs issued so far complete.
__device__ __forceinline__ void mma_commit_pair_if(uint32_t leader, uint64_t* bar) {
  asm volatile("{ .reg .pred q; setp.ne.b32 q, %1, 0; "
               "@q tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %2; }"
               ::"r"(smem_u32(bar)), "r"(leader), "h"(static_cast<uint16_t>(3)) : "memory");
}
// Arrive on a barrier of either CTA of the pair (`bar`: shared::cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Inverse of order_key (the key of -0 is the key of +0: it returns +0).
__device__ __forceinline__ float key_value(uint32_t key) {
  if (key == 0xFFFFFFFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// A float threshold t with {x : !(x < t)} = {x : order_key(x) >= P} when P is the key of
// a number; for a key in the range no number maps to (above +inf's key) it is +inf,
// which selects {order_key(x) >= order_key(+inf)}: a larger set, still of the same form.
// NaN logits always pass (their key is the largest).
__device__ __forceinline__ float pivot_threshold(uint32_t P) {
  const float t = key_value(P);
  return (t != t && P >= 0x80000000u) ? __int_as_float(0x7f800000) : t;
}

// One unit of a GEMM pass: an LM-head tile, a chunk of up to 512 hidden rows, and a
// range of 64-wide chunks of d (all of d unless the sample pass is split).
struct LmUnit {
  int tile, m0, mrows, kbeg, kend;
};
__device__ __forceinline__ LmUnit lm_unit(const LmParams& p, int u, int mchunks, int C, int crank, int nk) {
  const int kp = u % p.ksplit, rest = u / p.ksplit;
  LmUnit x;
  x.m0 = (rest % mchunks) * 512;
  x.tile = (rest / mchunks) * C + crank;
  x.mrows = min(512, p.M - x.m0);
  x.kbeg = kp * nk / p.ksplit;
  x.kend = (kp + 1) * nk / p.ksplit;
  return x;
}

}  // namespace

// MODE 0: sample pass (rows r * stride of the LM head, logits stored); MODE 1: filter
// pass (every row, logits at or above the row's pivot appended to its list).
//
// Launched as clusters of two CTAs that run one MMA of M = 256 together (tcgen05
// cta_group::2): CTA rank c of the pair stages its own 128-row LM-head tile (A rows
// 128c..) and half of each hidden-row part (B split along N), and its tensor memory
// receives its tile's 128 x N accumulators. Rank 0 issues the MMAs; both CTAs' copies
// count their bytes on rank 0's stage barrier, rank 0's commits release the stage in
// both CTAs, and both CTAs' epilogue warps release the accumulator on rank 0's barrier.
template <int MODE>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_gemm_kernel(const __grid_constant__ LmParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int NS = lm_stages(p.M);
  const uint32_t stage_bytes = static_cast<uint32_t>(lm_stage_bytes(p.M));
  const int h0 = lm_box0(p.M), h1 = lm_box1(p.M);  // hidden rows per CTA in parts 0 and 1
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + NS * stage_bytes);
  uint64_t* full = mbar;                     // [NS] rank 0: 1 arrival + both CTAs' bytes
  uint64_t* empty = mbar + NS;               // [NS] 1 commit (multicast by rank 0)
  uint64_t* dfull = mbar + 2 * NS;           // 1 commit (multicast by rank 0)
  uint64_t* dempty = mbar + 2 * NS + 1;      // rank 0: the epilogue warps of both CTAs
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(mbar + 2 * kLmMaxStages + 2);
  volatile int* fail = reinterpret_cast<volatile int*>(tbase_s + 1);
  float* thr_s = reinterpret_cast<float*>(smem + NS * stage_bytes + 128);  // [epilogue warp][4 x 32]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int crank = static_cast<int>(cluster_rank());
  const bool lead = crank == 0;
  const int cid = static_cast<int>(cluster_id());
  const int ncl = static_cast<int>(cluster_count());
  const int64_t rows = MODE == 0 ? p.S : p.V;                       // LM-head rows of this pass
  const int tiles = static_cast<int>((rows + kLmTile - 1) / kLmTile);
  const int groups = (tiles + 1) / 2;                               // tile pairs
  const int mchunks = (p.M + 511) / 512;
  const int units = groups * mchunks * p.ksplit;                    // per pair
  const int nk = p.d / kLmChunk;

  if (tid == 0) {
    for (int b = 0; b < 2 * NS + 2; ++b) {
      const uint32_t cnt = b == 2 * NS + 1 ? static_cast<uint32_t>(2 * kLmEpiWarps) : 1u;
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&mbar[b])), "r"(cnt));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    *fail = 0;
  }
  if (warp == 0) {  // one warp of each CTA of the pair allocates, together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(tbase_s)), "r"(kLmTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any copy or arrival lands in them
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tbase_s;
  if (MODE == 0 && tid == 0) allow_next_pass();
  const CUtensorMap* amap = MODE == 0 ? &p.ws_map : &p.w_map;
  const uint32_t full0 = peer_addr(full, 0);      // rank 0's full[0]; full[s] is 8 s further
  const uint32_t dempty0 = peer_addr(dempty, 0);  // rank 0's dempty

  if (warp == 0) {
    // ------------------------------------------------------------ tensor-map copies
    const uint32_t leader = lane == 0;
    const uint32_t bytes = 2 * kLmAStageBytes + 2 * 128 * (h0 + h1);  // both CTAs' boxes
    int g = 0;  // global chunk counter
    for (int u = cid; u < units && !__any_sync(kFull, *fail); u += ncl) {
      const LmUnit w = lm_unit(p, u, mchunks, 2, crank, nk);
      const int tile = w.tile, m0 = w.m0;
      // the first chunks of this tile go to L2 now (the rest are prefetched as it runs)
      const uint32_t pf = leader && static_cast<int64_t>(tile) * kLmTile < rows;  // tile holds rows
      for (int kc = w.kbeg; kc < min(w.kend, w.kbeg + NS); ++kc) tma_prefetch_2d_if(pf, amap, kc * kLmChunk, tile * kLmTile);
      bool ok = true;
      for (int kc = w.kbeg; kc < w.kend; ++kc, ++g) {
        const int s = g % NS;
        if (g >= NS && (ok = !__any_sync(kFull, !mbar_wait(&empty[s], ((g / NS) - 1) & 1, p, fail))) == false) break;
        if (kc + NS < w.kend) tma_prefetch_2d_if(pf, amap, (kc + NS) * kLmChunk, tile * kLmTile);
        unsigned char* st = smem + s * stage_bytes;
        const uint32_t bar = full0 + 8u * static_cast<uint32_t>(s);
        if (lead)
          asm volatile(
              "{ .reg .pred q; setp.ne.b32 q, %2, 0; @q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1; }"
              ::"r"(smem_u32(&full[s])), "r"(bytes), "r"(leader) : "memory");
        tma_2d_pair_if(leader, st, amap, kc * kLmChunk, tile * kLmTile, bar);
        tma_2d_pair_if(leader, st + kLmAStageBytes, &p.h_map0, kc * kLmChunk, m0 + crank * h0, bar);
        if (h1 > 0)
          tma_2d_pair_if(leader, st + kLmAStageBytes + h0 * 128, &p.h_map1, kc * kLmChunk, m0 + 256 + crank * h1, bar);
      }
      if (!ok) break;
    }
    // the last stages were consumed (so their copies landed) before the CTA leaves (bounded)
    for (int s = 0; s < NS; ++s) {
      if (g - 1 - s < 0) continue;
      const int gl = g - 1 - s;
      const uint64_t t0 = globaltimer_ns();
      while (!__all_sync(kFull, mbar_try(&empty[gl % NS], (gl / NS) & 1)) &&
             !__any_sync(kFull, globaltimer_ns() - t0 >= p.timeout_ns)) {}
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue (rank 0)
    const uint32_t leader = lane == 0;
    const int n0 = 2 * h0, n1 = 2 * h1;
    int g = 0, un = 0, last = -1;
    if (lead) {
      for (int u = cid; u < units && !__any_sync(kFull, *fail); u += ncl, ++un) {
        const LmUnit w = lm_unit(p, u, mchunks, 2, crank, nk);
        if (un >= 1 && __any_sync(kFull, !mbar_wait<true>(dempty, (un - 1) & 1, p, fail))) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        bool ok = true;
        for (int kc = w.kbeg; kc < w.kend; ++kc, ++g) {
          const int s = g % NS;
          if (__any_sync(kFull, !mbar_wait(&full[s], (g / NS) & 1, p, fail))) { ok = false; break; }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint32_t a0 = smem_u32(smem + s * stage_bytes), b0 = a0 + kLmAStageBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sw128_desc(a0 + kk * 32);
            const uint32_t acc = (kc > w.kbeg || kk > 0) ? 1u : 0u;
            for (int part = 0; part < 2; ++part) {
              const int np = part == 0 ? n0 : n1;
              if (np == 0) continue;
              const uint64_t bd = sw128_desc(b0 + part * h0 * 128 + kk * 32);
              asm volatile(
                  "{ .reg .pred p, q; setp.ne.b32 p, %4, 0; setp.ne.b32 q, %5, 0; "
                  "@q tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p; }"
                  ::"r"(tmem + part * 256), "l"(ad), "l"(bd), "r"(bf16_idesc(2 * kLmTile, np)), "r"(acc), "r"(leader)
                  : "memory");
            }
          }
          mma_commit_pair_if(leader, &empty[s]);
        }
        if (!ok) break;
        mma_commit_pair_if(leader, dfull);
        last = un;
      }
      // before tensor memory and the stages go (bounded): the last unit's MMAs are done
      // and every stage's release has arrived
      const uint64_t t0 = globaltimer_ns();
      if (last >= 0)
        while (!__all_sync(kFull, mbar_try(dfull, last & 1)) && !__any_sync(kFull, globaltimer_ns() - t0 >= p.timeout_ns)) {}
      for (int s = 0; s < NS; ++s) {
        if (g - 1 - s < 0) continue;
        const int gl = g - 1 - s;
        while (!__all_sync(kFull, mbar_try(&empty[gl % NS], (gl / NS) & 1)) &&
               !__any_sync(kFull, globaltimer_ns() - t0 >= p.timeout_ns)) {}
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if (MODE == 1) wait_previous_kernel();       // the pivots and the reset list counters
    const int q = warp & 3;                    // tensor-memory lane quadrant
    const int cg = (warp - 2) >> 2;            // column group: 32-column steps cg, cg + 4, ...
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    int un = 0;
    for (int u = cid; u < units && !__any_sync(kFull, *fail); u += ncl, ++un) {
      const LmUnit w = lm_unit(p, u, mchunks, 2, crank, nk);
      const int tile = w.tile, m0 = w.m0, mrows = w.mrows;
      // this warp's column thresholds (step i: columns 32 cg + 128 i + j at thr_w[32 i + j]),
      // read before the accumulator is ready: a logit passes when !(x < threshold)
      float* thr_w = thr_s + 128 * (warp - 2);
      if (MODE == 1) {
        __syncwarp();  // the previous unit's thresholds are read
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 32 * cg + 128 * i + lane;
          thr_w[32 * i + lane] = c < mrows ? pivot_threshold(__ldg(p.pivot + m0 + c)) : __int_as_float(0x7f800000);
        }
        __syncwarp();
      }
      if (__any_sync(kFull, !mbar_wait(dfull, un & 1, p, fail))) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int64_t r = static_cast<int64_t>(tile) * kLmTile + 32 * q + lane;  // LM-head row of the pass
      const bool rvalid = r < rows;
      // filter pass: appends wait in a four-entry queue {column, key} (the row r is this
      // lane's) and are written after the accumulator is released
      uint64_t q0 = 0, q1 = 0, q2 = 0, q3 = 0;
      int nq = 0;
      auto flush = [&]() {
        const uint64_t e[4] = {q0, q1, q2, q3};
        uint32_t pos[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < nq) pos[i] = atomicAdd(p.cnt + static_cast<size_t>(m0 + static_cast<int>(e[i] >> 32)) * kLmCntStride, 1u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < nq && pos[i] < static_cast<uint32_t>(p.cap))
            p.list[static_cast<size_t>(m0 + static_cast<int>(e[i] >> 32)) * p.cap + pos[i]] =
                pack_best(static_cast<uint32_t>(e[i]), static_cast<uint32_t>(r));
        nq = 0;
      };
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c0 = 32 * cg + 128 * i;
        if (c0 >= mrows) break;
        // hidden row c0 + j sits in column c0 + j (part 1 starts at column 256)
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
            "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
              "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
            : "r"(tmem + lane_off + static_cast<uint32_t>(c0)) : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int ncol = min(32, mrows - c0);
        if constexpr (MODE == 0) {
          if (rvalid) {
            float* dst = p.sample + static_cast<size_t>(m0 + c0) * p.S + r;
            if (p.ksplit > 1) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < ncol) atomicAdd(dst + static_cast<size_t>(j) * p.S, __uint_as_float(v[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < ncol) dst[static_cast<size_t>(j) * p.S] = __uint_as_float(v[j]);
            }
          }
        } else {
          uint32_t pass = 0;
          const float4* t4 = reinterpret_cast<const float4*>(thr_w + 32 * i);
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 t = t4[j4];
            pass |= !(__uint_as_float(v[4 * j4 + 0]) < t.x) ? (1u << (4 * j4 + 0)) : 0u;
            pass |= !(__uint_as_float(v[4 * j4 + 1]) < t.y) ? (1u << (4 * j4 + 1)) : 0u;
            pass |= !(__uint_as_float(v[4 * j4 + 2]) < t.z) ? (1u << (4 * j4 + 2)) : 0u;
            pass |= !(__uint_as_float(v[4 * j4 + 3]) < t.w) ? (1u << (4 * j4 + 3)) : 0u;
          }
          if (!rvalid) pass = 0;
          pass &= ncol == 32 ? 0xFFFFFFFFu : ((1u << ncol) - 1u);
          while (pass) {
            const int j = __ffs(pass) - 1;
            pass &= pass - 1;
            // v[j] for a lane-dependent j: a five-level selection on the bits of j
            uint32_t x16[16], x8[8], x4[4], x2[2];
#pragma unroll
            for (int t = 0; t < 16; ++t) x16[t] = (j & 16) ? v[t + 16] : v[t];
#pragma unroll
            for (int t = 0; t < 8; ++t) x8[t] = (j & 8) ? x16[t + 8] : x16[t];
#pragma unroll
            for (int t = 0; t < 4; ++t) x4[t] = (j & 4) ? x8[t + 4] : x8[t];
#pragma unroll
            for (int t = 0; t < 2; ++t) x2[t] = (j & 2) ? x4[t + 2] : x4[t];
            const uint32_t x = (j & 1) ? x2[1] : x2[0];
            if (nq == 4) flush();
            q3 = q2; q2 = q1; q1 = q0;
            q0 = (static_cast<uint64_t>(c0 + j) << 32) | order_key(__uint_as_float(x));
            ++nq;
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(dempty0);  // rank 0's MMAs may overwrite the accumulator
      if (MODE == 1 && nq > 0) flush();
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (MODE == 1 && tid == 0) allow_next_pass();
  cluster_sync();  // no CTA leaves while its pair may still write into it or arrive on it
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kLmTmemCols) : "memory");
}

namespace {

constexpr int kSelThreads = 512;

// One radix-selection step, run by warp 0 of the block: from a 256-bin histogram of
// the items that share the current prefix, and the number of items above that prefix,
// the bin holding the `rank`-th largest item (1-based), the items above that bin, and
// whether the bin's items are exactly the ones still needed (then the selection ends:
// every item at or above the bin's lower edge is taken). Lane l scans bins
// 255 - 8l ... 248 - 8l after a warp prefix sum of the lanes' totals.
__device__ __forceinline__ void pick_bin(const int* hist, int above, int rank, int* sel) {
  const int lane = threadIdx.x & 31;
  int c[8], tot = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = hist[255 - 8 * lane - i];
    tot += c[i];
  }
  int incl = tot;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, off);
    if (lane >= off) incl += y;
  }
  const int excl = incl - tot;
  if (above + excl < rank && rank <= above + incl) {
    int acc = above + excl;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (acc + c[i] >= rank) {
        sel[0] = 255 - 8 * lane - i;
        sel[1] = acc;
        sel[2] = acc + c[i] == rank;
        break;
      }
      acc += c[i];
    }
  }
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ int high_bit(uint64_t x) { return 63 - __clzll(static_cast<long long>(x)); }

// Block-wide radix selection over the n words (uint32_t or uint64_t) in shared memory:
// returns T with at least `rank` words >= T and, when the words are distinct, exactly
// `rank`. The digits start at the highest bit where the smallest and largest word differ
// (the bits above are common to all words and need no pass), eight bits a pass, and the
// selection stops as soon as a bin holds exactly the words still needed. `hist` [256],
// `sel` [3] and `mm` [2] are shared scratch; every thread of the block calls it.
template <typename W>
__device__ W block_select(const W* words, int n, int rank, int* hist, int* sel, unsigned long long* mm) {
  constexpr int kBits = 8 * sizeof(W);
  uint64_t lo = ~0ull, hi = 0ull;
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    const uint64_t w = words[t];
    lo = w < lo ? w : lo;
    hi = w > hi ? w : hi;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t a = shfl_xor64(lo, o), b = shfl_xor64(hi, o);
    lo = a < lo ? a : lo;
    hi = b > hi ? b : hi;
  }
  if (threadIdx.x == 0) { mm[0] = ~0ull; mm[1] = 0ull; }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&mm[0], static_cast<unsigned long long>(lo));
    atomicMax(&mm[1], static_cast<unsigned long long>(hi));
  }
  __syncthreads();
  lo = mm[0];
  hi = mm[1];
  __syncthreads();
  if (lo == hi) return static_cast<W>(lo);
  int top = high_bit(lo ^ hi);                  // highest bit that differs
  uint64_t prefix = top + 1 < kBits ? (lo >> (top + 1)) : 0ull;  // common bits above it
  int above = 0, low = 0;
  while (top >= 0) {
    low = top >= 7 ? top - 7 : 0;
    const int width = top - low + 1;
    const uint64_t mask = (1ull << width) - 1ull;
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    if (threadIdx.x == 0) { sel[0] = 0; sel[1] = above; sel[2] = 1; }
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
      const uint64_t w = words[t];
      const uint64_t up = top + 1 < kBits ? (w >> (top + 1)) : 0ull;
      if (up == prefix) atomicAdd(&hist[static_cast<int>((w >> low) & mask)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) pick_bin(hist, above, rank, sel);
    __syncthreads();
    prefix = (prefix << width) | static_cast<uint64_t>(sel[0]);
    above = sel[1];
    const bool done = sel[2] != 0;
    __syncthreads();
    if (done) break;
    top = low - 1;
  }
  return static_cast<W>(prefix << low);
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

// Per hidden row: the pivot P, a key with at least j of the row's sampled keys at or
// above it (the j-th largest, or the lower edge of a radix bin holding exactly the keys
// still needed), by a block radix selection over the keys staged in shared memory (one
// CTA per row); the row's list counter is zeroed. Rows of more than kPivotSmemKeys
// samples use their first kPivotSmemKeys with j scaled alike (the pivot only steers the
// list's size; the list itself is exact).
constexpr int kPivotSmemKeys = 40960;

__global__ void __launch_bounds__(kSelThreads) lmhead_pivot_kernel(const LmParams p, int j) {
  extern __shared__ __align__(16) uint32_t keys_s[];
  __shared__ int hist[256];
  __shared__ int sel[3];
  __shared__ unsigned long long mm[2];
  if (threadIdx.x == 0) allow_next_pass();
  wait_previous_kernel();  // the sampled logits
  const int m = blockIdx.x;
  const float* x = p.sample + static_cast<size_t>(m) * p.S;
  const int n = p.S < kPivotSmemKeys ? p.S : kPivotSmemKeys;
  int rank = n == p.S ? j : static_cast<int>((static_cast<int64_t>(j) * n) / p.S);
  rank = rank < 1 ? 1 : (rank > n ? n : rank);
  for (int s0 = threadIdx.x; s0 < n; s0 += 8 * blockDim.x) {
    float xv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = s0 + i * blockDim.x;
      xv[i] = s < n ? x[s] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = s0 + i * blockDim.x;
      if (s < n) keys_s[s] = order_key(xv[i]);
    }
  }
  __syncthreads();
  const uint32_t P = block_select<uint32_t>(keys_s, n, rank, hist, sel, mm);
  if (threadIdx.x == 0) {
    p.pivot[m] = P;
    p.cnt[static_cast<size_t>(m) * kLmCntStride] = 0u;
  }
}

// Per hidden row: the k largest packed words of its list (one CTA per row, the list read
// from L2, block radix selection), or the exact path over the whole row when the list is
// short, overflowed or the fallback is forced.
__global__ void __launch_bounds__(kSelThreads) lmhead_select_kernel(const LmParams p) {
  __shared__ int hist[256];
  __shared__ int sel[3];
  __shared__ unsigned long long mm[2];
  __shared__ int outpos;
  wait_previous_kernel();  // the lists and their counters
  const int m = blockIdx.x;
  const int k = p.k;
  const uint32_t n_all = p.cnt[static_cast<size_t>(m) * kLmCntStride];
  const bool exact = (p.flags & kLmForceExact) || n_all < static_cast<uint32_t>(k) ||
                     n_all > static_cast<uint32_t>(p.cap);
  int32_t* cand = p.cand + static_cast<size_t>(m) * k;
  float* cbase = p.cand_base + static_cast<size_t>(m) * k;
  if (threadIdx.x == 0) outpos = 0;
  if (!exact) {
    const int n = static_cast<int>(n_all);
    const uint64_t* words = p.list + static_cast<size_t>(m) * p.cap;  // read where the filter pass left them (L2)
    const uint64_t thr = block_select<uint64_t>(words, n, k, hist, sel, mm);
    // words are distinct (one per vocabulary entry): exactly k are >= the threshold,
    // written in list order (positions by a warp ballot and one shared add per warp)
    for (int t0 = threadIdx.x & ~31; t0 < n; t0 += blockDim.x) {
      const int t = t0 + (threadIdx.x & 31);
      const uint64_t w = t < n ? words[t] : 0ull;
      const bool take = t < n && w >= thr;
      const uint32_t ball = __ballot_sync(kFull, take);
      int base = 0;
      if ((threadIdx.x & 31) == 0 && ball) base = atomicAdd(&outpos, __popc(ball));
      base = __shfl_sync(kFull, base, 0);
      if (take) {
        const int pos = base + __popc(ball & ((1u << (threadIdx.x & 31)) - 1u));
        cand[pos] = unpack_idx(w);
        cbase[pos] = key_value(static_cast<uint32_t>(w >> 32));
      }
    }
    return;
  }
  if (threadIdx.x == 0 && p.stats) {  // every exact-path row, and separately the overflowed ones
    atomicAdd(p.stats, 1);
    if (n_all > static_cast<uint32_t>(p.cap)) atomicAdd(p.stats + 1, 1);
  }
  // exact path: radix selection of the k-th largest key over the whole recomputed row,
  // then an index-ordered pass taking keys above it and the first ties
  uint32_t prefix = 0;
  int above = 0, sh = 0;
  bool all_of_bin = false;
  for (int pass = 0; pass < 4; ++pass) {
    sh = 24 - 8 * pass;
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    if (threadIdx.x == 0) { sel[0] = 0; sel[1] = above; sel[2] = 1; }
    __syncthreads();
    for (int64_t v = threadIdx.x; v < p.V; v += blockDim.x) {
      const uint32_t key = order_key(dot_row(p, m, v));
      if (pass == 0 || (key >> (sh + 8)) == prefix) atomicAdd(&hist[(key >> sh) & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) pick_bin(hist, above, k, sel);
    __syncthreads();
    prefix = (prefix << 8) | static_cast<uint32_t>(sel[0]);
    above = sel[1];
    all_of_bin = sel[2] != 0;
    __syncthreads();
    if (all_of_bin) break;
  }
  // all_of_bin: every key >= thr is taken (exactly k). Otherwise thr is the k-th largest
  // key and the first k - above of the keys equal to it, in index order, are taken.
  const uint32_t thr = prefix << sh;
  const int need_eq = all_of_bin ? 0 : k - above;
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
    const bool take = (v < p.V) && (all_of_bin ? key >= thr : (key > thr || (eq && before < need_eq)));
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


namespace {

// Grid of a GEMM pass: CTA pairs (clusters of two), no more than can be resident at once
// (one CTA per SM) and no more than there are pair steps of work.
template <int MODE>
cudaError_t launch_gemm(LmParams& p, int sms, size_t smem, int units, cudaStream_t stream) {
  auto fn = lmhead_gemm_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the filter pass follows the pivot pass as a programmatic dependent; the sample pass
  // starts the call in plain stream order (it reads the caller's inputs)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kLmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = MODE == 1 ? 2 : 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (sms / 2)));
  int max_clusters = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg)) != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min(max_clusters, std::max(1, units))));
  return cudaLaunchKernelEx(&cfg, fn, p);
}

// The pivot and select passes: one CTA per hidden row, launched as programmatic
// dependents of the pass before them.
template <typename... Args>
cudaError_t launch_dependent(void (*fn)(Args...), unsigned grid, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

}  // namespace

cudaError_t launch_lmhead(LmParams& p, int sms, int pivot_rank, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(lm_gemm_smem(p.M));
  cudaError_t e;
  const size_t psmem = static_cast<size_t>(std::min(p.S, kPivotSmemKeys)) * 4;
  if ((e = cudaFuncSetAttribute(lmhead_pivot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPivotSmemKeys * 4)) != cudaSuccess)
    return e;
  const int mchunks = (p.M + 511) / 512;
  const int units0 = static_cast<int>(((p.S + kLmTile - 1) / kLmTile + 1) / 2) * mchunks;  // pair steps
  const int units1 = static_cast<int>(((p.V + kLmTile - 1) / kLmTile + 1) / 2) * mchunks;
  // the sample pass has few tiles: split d so that every cluster has work, the parts
  // summed by fp32 atomics into the zeroed sample rows (the pivot needs no exact sums)
  const int nk = p.d / kLmChunk;
  p.ksplit = std::max(1, std::min(std::min(nk, 8), (sms / 2) / std::max(1, units0)));
  if (p.ksplit > 1 &&
      (e = cudaMemsetAsync(p.sample, 0, static_cast<size_t>(p.M) * p.S * sizeof(float), stream)) != cudaSuccess)
    return e;
  if ((e = launch_gemm<0>(p, sms, smem, units0 * p.ksplit, stream)) != cudaSuccess) return e;
  p.ksplit = 1;
  if ((e = launch_dependent(lmhead_pivot_kernel, static_cast<unsigned>(p.M), psmem, stream, p, pivot_rank)) !=
      cudaSuccess)
    return e;
  if ((e = launch_gemm<1>(p, sms, smem, units1, stream)) != cudaSuccess) return e;
  return launch_dependent(lmhead_select_kernel, static_cast<unsigned>(p.M), 0, stream, p);
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
