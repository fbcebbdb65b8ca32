// Full-vocabulary Markov draft walk on CUDA cores: one persistent cooperative kernel
// for all K draft positions (vLLM PR #62958, "Overview": the whole walk in one
// cooperative kernel, W2 mostly resident in shared memory, the rest streamed from L2,
// one packed atomic per step for the cross-CTA argmax).
//
// Work split. CTA c owns the contiguous vocabulary slice [c*V/G, (c+1)*V/G). The first
// `resident_rows` rows of the slice are copied into shared memory while draft position
// 0 streams them from HBM, and are read from shared memory at every later position.
// Of the remaining rows, each warp keeps its first 32-row blocks (int8: two, bf16: one)
// in tensor memory, which this kernel otherwise leaves idle: written at the first pass
// and read back (tcgen05.ld) at every later one. The rest are re-read from L2.
//
// Contraction. Eight lanes share one W2 row; lane j owns the 16-byte chunks j, j+8
// (int8: 32 values) or j, j+8, j+16, j+24 (bf16: 32 values) of every row, so the
// embedding slice it multiplies with stays in registers. Each 8-lane group handles 8
// rows at a time and a 3-stage xor butterfly leaves lane j with the total of row j.
//   * int8 W2: the embedding row e is scaled by a power of two 2^s to a 24-bit
//     integer and split into one signed and two unsigned byte limbs; dp4a then gives
//     the exact integer sum_k q[v,k] * round(e_k 2^s), and the bias is
//     scale_v * 2^-s * sum. bf16 e has 8 significant bits, so every entry within
//     2^16 of max|e| is represented exactly; the result is at least as accurate as an
//     fp32 accumulation and is independent of summation order.
//   * bf16 W2: fp32 FMA in a fixed order (lane-local k order, then the butterfly),
//     identical for every row, so identical rows give identical bias values.
//
// Per-position cross-CTA argmax: each CTA reduces its (orderable key, first index)
// word per request row, issues one 64-bit atomicMax into slot[i][b], and the grid
// meets at a bounded barrier; then every CTA reads the winning token.
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "walk_params.cuh"

namespace dspark {

namespace {

__device__ __forceinline__ int dp4a_ss(int a, int b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_su(int a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Reduce-scatter of 8 per-row partials over the 8 lanes of a group: afterwards lane
// j (j = lane & 7) holds the sum over the group of partial j in v[0]. Every row's
// sum is formed by the same pairing tree (commutative adds only), so identical rows
// give identical results.
template <typename T>
__device__ __forceinline__ T butterfly8(T (&v)[8], int lane) {
  const bool u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const T send = u4 ? v[t] : v[t + 4];
    const T keep = u4 ? v[t + 4] : v[t];
    v[t] = keep + __shfl_xor_sync(kFull, send, 4);
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const T send = u2 ? v[t] : v[t + 2];
    const T keep = u2 ? v[t + 2] : v[t];
    v[t] = keep + __shfl_xor_sync(kFull, send, 2);
  }
  const T send = u1 ? v[0] : v[1];
  const T keep = u1 ? v[1] : v[0];
  return keep + __shfl_xor_sync(kFull, send, 1);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most `pending` of this thread's most recent commit groups are in flight.
__device__ __forceinline__ void cp_async_wait(int pending) {
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

__device__ __forceinline__ uint4 ld_row_chunk(const unsigned char* row_global, int chunk) {
  return __ldg(reinterpret_cast<const uint4*>(row_global) + chunk);
}

// x * 2^s for |s| <= 252 as two exact multiplies by normal powers of two.
__device__ __forceinline__ float pow2_lo(int s) { return __int_as_float((s / 2 + 127) << 23); }
__device__ __forceinline__ float pow2_hi(int s) { return __int_as_float((s - s / 2 + 127) << 23); }
__device__ __forceinline__ float mul_pow2(float x, int s) {
  return __fmul_rn(__fmul_rn(x, pow2_lo(s)), pow2_hi(s));
}

// Limbs of the 16 integers of one chunk: hi (signed byte), mid and lo (unsigned).
struct Limbs {
  int hi[4];
  uint32_t mid[4], lo[4];
};

// Limb words of one embedding row: [3][64] uint32, word w of limb j packs the byte j
// of the 24-bit integers round(e_k 2^shift) for k = 4w .. 4w+3.
__device__ __forceinline__ void load_limbs(const uint32_t* limb_row, int chunk, Limbs& L) {
  const uint4 h = reinterpret_cast<const uint4*>(limb_row)[chunk];
  const uint4 m = reinterpret_cast<const uint4*>(limb_row + 64)[chunk];
  const uint4 l = reinterpret_cast<const uint4*>(limb_row + 128)[chunk];
  L.hi[0] = static_cast<int>(h.x); L.hi[1] = static_cast<int>(h.y);
  L.hi[2] = static_cast<int>(h.z); L.hi[3] = static_cast<int>(h.w);
  L.mid[0] = m.x; L.mid[1] = m.y; L.mid[2] = m.z; L.mid[3] = m.w;
  L.lo[0] = l.x; L.lo[1] = l.y; L.lo[2] = l.z; L.lo[3] = l.w;
}

__device__ __forceinline__ void dot_int8_chunk(const uint4& q, const Limbs& L, int& h, int& m,
                                               int& l) {
  const int qw[4] = {static_cast<int>(q.x), static_cast<int>(q.y), static_cast<int>(q.z),
                     static_cast<int>(q.w)};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    h = dp4a_ss(qw[w], L.hi[w], h);
    m = dp4a_su(qw[w], L.mid[w], m);
    l = dp4a_su(qw[w], L.lo[w], l);
  }
}

__device__ __forceinline__ float dot_int8_chunk_f32(const uint4& q, const float* e, float acc) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int w = 0; w < 4; ++w)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int qi = static_cast<int>(static_cast<int8_t>((qw[w] >> (8 * t)) & 0xFFu));
      acc = __fmaf_rn(static_cast<float>(qi), e[4 * w + t], acc);
    }
  return acc;
}

__device__ __forceinline__ float dot_bf16_chunk(const uint4& q, const float* e, float acc) {
  const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    acc = __fmaf_rn(bf16_lo(qw[w]), e[2 * w], acc);
    acc = __fmaf_rn(bf16_hi(qw[w]), e[2 * w + 1], acc);
  }
  return acc;
}

// Score of one vocabulary entry and its argmax word. sampled / T: row b's settings.
template <bool PROB, bool LOGITS>
__device__ __forceinline__ uint64_t score_entry(const WalkParams& p, int b, int i, int64_t v,
                                                float base_v, float bias, uint64_t seed,
                                                bool sampled, float T) {
  const size_t o = (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v;
  const float l = __fadd_rn(base_v, bias);
  if (LOGITS) p.logits[o] = f32_to_bf16_bits(l);
  float s = l;
  if (PROB && sampled) {
    const float lb = bf16_to_f32(f32_to_bf16_bits(l));
    const float x = T == 1.0f ? lb : __fdiv_rn(lb, T);
    const uint4 w = philox_block(seed, b, i, static_cast<uint32_t>(v >> 2));
    s = __fadd_rn(x, gumbel_from_word(uint4_get(w, static_cast<int>(v & 3))));
  }
  return pack_best(order_key(s), static_cast<uint32_t>(v));
}

// One W2 row's chunks of this lane (int8: 2, bf16: 4 x 16 bytes) to / from tensor
// memory: 8 or 16 consecutive 32-bit columns of the lane's own row of tensor memory.
template <int C>
__device__ __forceinline__ void tmem_st_chunks(uint32_t taddr, const uint4 (&q)[C]);
template <>
__device__ __forceinline__ void tmem_st_chunks<2>(uint32_t taddr, const uint4 (&q)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               ::"r"(taddr), "r"(q[0].x), "r"(q[0].y), "r"(q[0].z), "r"(q[0].w), "r"(q[1].x), "r"(q[1].y),
                 "r"(q[1].z), "r"(q[1].w) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_chunks<4>(uint32_t taddr, const uint4 (&q)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
               "%11, %12, %13, %14, %15, %16};"
               ::"r"(taddr), "r"(q[0].x), "r"(q[0].y), "r"(q[0].z), "r"(q[0].w), "r"(q[1].x), "r"(q[1].y),
                 "r"(q[1].z), "r"(q[1].w), "r"(q[2].x), "r"(q[2].y), "r"(q[2].z), "r"(q[2].w), "r"(q[3].x),
                 "r"(q[3].y), "r"(q[3].z), "r"(q[3].w) : "memory");
}
template <int C>
__device__ __forceinline__ void tmem_ld_chunks(uint32_t taddr, uint4 (&q)[C]);
template <>
__device__ __forceinline__ void tmem_ld_chunks<2>(uint32_t taddr, uint4 (&q)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(q[0].x), "=r"(q[0].y), "=r"(q[0].z), "=r"(q[0].w), "=r"(q[1].x), "=r"(q[1].y),
                 "=r"(q[1].z), "=r"(q[1].w) : "r"(taddr) : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
template <>
__device__ __forceinline__ void tmem_ld_chunks<4>(uint32_t taddr, uint4 (&q)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
               "%11, %12, %13, %14, %15}, [%16];"
               : "=r"(q[0].x), "=r"(q[0].y), "=r"(q[0].z), "=r"(q[0].w), "=r"(q[1].x), "=r"(q[1].y),
                 "=r"(q[1].z), "=r"(q[1].w), "=r"(q[2].x), "=r"(q[2].y), "=r"(q[2].z), "=r"(q[2].w),
                 "=r"(q[3].x), "=r"(q[3].y), "=r"(q[3].z), "=r"(q[3].w) : "r"(taddr) : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace

template <bool INT8, bool PROB, bool LOGITS>
__global__ void __launch_bounds__(kWalkThreads, 1) walk_cc_kernel(const WalkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kRowBytes = INT8 ? kRank : 2 * kRank;
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j8 = lane & 7, grp = lane >> 3;

  const int64_t v0 = static_cast<int64_t>(cta) * p.V / G;
  const int64_t v1 = static_cast<int64_t>(cta + 1) * p.V / G;
  const int n = static_cast<int>(v1 - v0);
  const int res = min(p.resident_rows, n & ~31);

  // Shared memory: resident W2 rows | scales of the slice (int8) | embedding rows |
  // shifts | previous tokens | per-row CTA argmax words | reduction scratch | flag.
  unsigned char* w2s = smem;
  float* scale_s = reinterpret_cast<float*>(smem + static_cast<size_t>(p.resident_rows) * kRowBytes);
  uint16_t* e_s = reinterpret_cast<uint16_t*>(scale_s + (INT8 ? p.slice_cap : 0));
  uint32_t* limb_s = reinterpret_cast<uint32_t*>(e_s + static_cast<size_t>(p.bs) * kRank);
  int* sh_shift = reinterpret_cast<int*>(limb_s + (INT8 ? static_cast<size_t>(p.bs) * 3 * 64 : 0));
  int* prev_s = sh_shift + 64;
  uint64_t* best_s = reinterpret_cast<uint64_t*>(prev_s + 64);
  uint64_t* red = best_s + 64;
  int* flag = reinterpret_cast<int*>(red + kWalkWarps);
  uint32_t* tbase_s = reinterpret_cast<uint32_t*>(flag + 1);  // tensor-memory base address

  const unsigned char* w2g = INT8 ? reinterpret_cast<const unsigned char*>(p.w2q)
                                  : reinterpret_cast<const unsigned char*>(p.w2);
  w2g += static_cast<size_t>(v0) * kRowBytes;

  const bool skip0 = (p.sync.flags & DSPARK_FLAG_SKIP_ARRIVAL_CTA0) && cta == 0;

  for (int t = threadIdx.x; t < p.bs; t += blockDim.x) {
    const int32_t tok = p.prev[t];
    const bool ok = tok >= 0 && static_cast<int64_t>(tok) < p.V;
    const bool settings = row_settings_ok(p, PROB, t);
    prev_s[t] = ok && settings ? tok : -1;
    if (!ok && cta == 0) report(p.sync.status_dev, DSPARK_ERR_BAD_TOKEN);
    if (!settings && cta == 0) report(p.sync.status_dev, DSPARK_ERR_INVALID_ARG);
  }
  if (INT8)
    for (int r = threadIdx.x; r < n; r += blockDim.x) scale_s[r] = __ldg(p.scales + v0 + r);
  // Base logits of the first two positions towards L2; later positions are fetched
  // two steps ahead, so the epilogue's loads hit L2 instead of cold HBM.
  prefetch_base_slice(p, v0, n, 0);
  prefetch_base_slice(p, v0, n, 1);
  bool filled = false;

  // Tensor memory (all 512 columns, idle otherwise in this kernel) keeps the first
  // kTmBlocks of each warp's 32-row blocks beyond the resident rows, written at the
  // walk's first pass over them and read back at every later one instead of from L2.
  // Warp w owns the lanes of quadrant w % 4 and columns 128 (w / 4) .. + 127.
  constexpr int kChunksPerRow = INT8 ? 2 : 4;
  constexpr int kTmBlocks = 128 / (8 * kChunksPerRow * 4);  // blocks per warp: int8 2, bf16 1
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;"
                 ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(tbase_s))) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm_warp = *tbase_s + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 128u * (warp >> 2);
  auto release_tmem = [&]() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(*tbase_s) : "memory");
  };

  for (int i = 0; i < p.K; ++i) {
    __syncthreads();
    // Markov embeddings of the previous tokens (bf16 rows into shared memory) and,
    // for int8 W2, the power-of-two shift that makes each row a 24-bit integer vector.
    for (int b = warp; b < p.bs; b += kWalkWarps) {
      const int tok = prev_s[b];
      float amax = 0.f;
      if (tok >= 0) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(tok) * kRank) + lane);
        reinterpret_cast<uint4*>(e_s + static_cast<size_t>(b) * kRank)[lane] = w;
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          amax = fmaxf(amax, fabsf(bf16_lo(ww[t])));
          amax = fmaxf(amax, fabsf(bf16_hi(ww[t])));
          if (!isfinite(bf16_lo(ww[t])) || !isfinite(bf16_hi(ww[t]))) amax = __int_as_float(0x7F800000);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
      int shift = 0;
      if (!isfinite(amax)) {
        shift = 1 << 30;  // marks a non-finite embedding row: fp32 fallback
      } else if (amax > 0.f) {
        int ex;
        frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)
        shift = 23 - ex;    // amax * 2^shift in [2^22, 2^23)
      }
      if (lane == 0) sh_shift[b] = shift;
      if (INT8 && tok >= 0 && shift != (1 << 30)) {
        // This lane's 8 values k = 8 lane .. 8 lane + 7 become two words per limb.
        const uint4 w = reinterpret_cast<const uint4*>(e_s + static_cast<size_t>(b) * kRank)[lane];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        uint32_t hl[2] = {0u, 0u}, ml[2] = {0u, 0u}, ll[2] = {0u, 0u};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float x = (t & 1) ? bf16_hi(ww[t >> 1]) : bf16_lo(ww[t >> 1]);
          const int xi = __float2int_rn(mul_pow2(x, shift));
          const int wsel = t >> 2, sh8 = 8 * (t & 3);
          hl[wsel] |= (static_cast<uint32_t>(xi >> 16) & 0xFFu) << sh8;
          ml[wsel] |= (static_cast<uint32_t>(xi >> 8) & 0xFFu) << sh8;
          ll[wsel] |= (static_cast<uint32_t>(xi) & 0xFFu) << sh8;
        }
        uint32_t* lr = limb_s + static_cast<size_t>(b) * 3 * 64;
        reinterpret_cast<uint2*>(lr)[lane] = make_uint2(hl[0], hl[1]);
        reinterpret_cast<uint2*>(lr + 64)[lane] = make_uint2(ml[0], ml[1]);
        reinterpret_cast<uint2*>(lr + 128)[lane] = make_uint2(ll[0], ll[1]);
      }
    }
    __syncthreads();

    for (int b = 0; b < p.bs; ++b) {
      if (prev_s[b] < 0) continue;  // uniform over the CTA
      const bool sampled = row_sampled(p, PROB, b);
      const float T_b = sampled ? row_temperature(p, b) : 1.0f;
      const uint64_t seed = sampled ? p.seeds[b] : 0ull;
      const uint16_t* eb = e_s + static_cast<size_t>(b) * kRank;
      const int shift = sh_shift[b];
      const bool float_path = INT8 && shift == (1 << 30);
      const bool fill = !filled;

      const float inv_lo = pow2_lo(-shift), inv_hi = pow2_hi(-shift);

      // The row loop, instantiated once with the integer limbs (int8 W2, finite
      // embedding) and once with fp32 embedding values (bf16 W2, or the fallback for a
      // non-finite embedding row), so each instance keeps only its own registers.
      auto row_loop = [&](auto use_limbs_tag) -> uint64_t {
        constexpr bool LIMBS = decltype(use_limbs_tag)::value;
        Limbs LA, LB;
        float ef[LIMBS ? 1 : 32];
        if constexpr (LIMBS) {
          const uint32_t* lr = limb_s + static_cast<size_t>(b) * 3 * 64;
          load_limbs(lr, j8, LA);
          load_limbs(lr, j8 + 8, LB);
        } else {
          constexpr int cw = INT8 ? 16 : 8;  // values per chunk
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int chunk = j8 + 8 * (c / cw);
            ef[c] = bf16_to_f32(eb[chunk * cw + (c % cw)]);
          }
        }
        uint64_t best = 0ull;
        // Warp w owns the 32-row blocks w, w + 16, ... of the slice. Blocks that are
        // re-read from L2 every step (beyond the resident rows) come first so their
        // latency overlaps the other warps' shared-memory blocks.
        const int nblk = n > 32 * warp ? (n - 32 * warp + 32 * kWalkWarps - 1) / (32 * kWalkWarps) : 0;
        int nres_blk = 0;  // the warp's resident blocks are its first nres_blk blocks
        while (nres_blk < nblk && 32 * warp + 32 * kWalkWarps * nres_blk + 32 <= res) ++nres_blk;
        // Position 0 brings the resident blocks in with asynchronous copies (one commit
        // group per block, each lane copying exactly the chunks it reads later).
        const bool fill_now = fill && i == 0;
        if (fill_now) {
          for (int t = 0; t < nres_blk; ++t) {
            const int rb = 32 * warp + 32 * kWalkWarps * t + 8 * grp;
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
#pragma unroll
              for (int c = 0; c < kRowBytes / 128; ++c) {
                const size_t off = static_cast<size_t>(rb + rr) * kRowBytes + 16 * (j8 + 8 * c);
                cp_async16(w2s + off, w2g + off);
              }
            cp_async_commit();
          }
        }
        auto block_r0 = [&](int k) {  // k-th block in processing order
          const int t = k < nblk - nres_blk ? nres_blk + k : k - (nblk - nres_blk);
          return 32 * warp + 32 * kWalkWarps * t;
        };
        auto load_base = [&](int r) {
          return r < n ? bf16_to_f32(__ldg(p.base + (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v0 + r))
                       : 0.f;
        };
        float base_next = nblk > 0 ? load_base(block_r0(0) + 8 * grp + j8) : 0.f;
        for (int k = 0; k < nblk; ++k) {
          const int r0 = block_r0(k);
          const bool resident = r0 + 32 <= res;
          const bool from_smem = resident && (i > 0 || !fill || fill_now);
          const bool store_smem = false;
          // streamed blocks come first: block k < kTmBlocks of them lives in tensor memory
          const bool in_tm = !resident && k < kTmBlocks;
          const bool tm_store = in_tm && fill, tm_load = in_tm && !fill;
          const uint32_t tm_blk = tm_warp + static_cast<uint32_t>(k) * (8 * kChunksPerRow * 4);
          if (fill_now && resident) cp_async_wait(nblk - 1 - k);
          const int rbase = r0 + 8 * grp;
          // The lane's own epilogue row: its base logit was loaded one block ahead.
          const int r_out = rbase + j8;
          const float base_v = base_next;
          if (k + 1 < nblk) base_next = load_base(block_r0(k + 1) + 8 * grp + j8);
          [[maybe_unused]] const float scale_v = (INT8 && r_out < n) ? scale_s[r_out] : 0.f;
          float fpart[8];
          int hpart[8], mpart[8];
#pragma unroll
          for (int rr = 0; rr < 8; ++rr) {
            const int r = rbase + rr;
            constexpr int kChunks = INT8 ? 2 : 4;
            uint4 q[kChunks];
            if (tm_load) {
              tmem_ld_chunks<kChunks>(tm_blk + rr * (kChunks * 4), q);
            } else {
#pragma unroll
              for (int c = 0; c < kChunks; ++c) {
                if (r < n) {
                  if (from_smem)
                    q[c] = reinterpret_cast<const uint4*>(w2s + static_cast<size_t>(r) * kRowBytes)[j8 + 8 * c];
                  else
                    q[c] = ld_row_chunk(w2g + static_cast<size_t>(r) * kRowBytes, j8 + 8 * c);
                  if (store_smem)
                    reinterpret_cast<uint4*>(w2s + static_cast<size_t>(r) * kRowBytes)[j8 + 8 * c] = q[c];
                } else {
                  q[c] = make_uint4(0u, 0u, 0u, 0u);
                }
              }
              if (tm_store) tmem_st_chunks<kChunks>(tm_blk + rr * (kChunks * 4), q);
            }
            if constexpr (LIMBS) {
              int h = 0, m = 0, l = 0;
              dot_int8_chunk(q[0], LA, h, m, l);
              dot_int8_chunk(q[1], LB, h, m, l);
              hpart[rr] = h;
              mpart[rr] = m * 256 + l;
            } else if constexpr (INT8) {
              float a = 0.f;
              a = dot_int8_chunk_f32(q[0], ef, a);
              a = dot_int8_chunk_f32(q[1], ef + 16, a);
              fpart[rr] = a;
            } else {
              float a = 0.f;
#pragma unroll
              for (int c = 0; c < kChunks; ++c) a = dot_bf16_chunk(q[c], ef + 8 * c, a);
              fpart[rr] = a;
            }
          }
          if (tm_store) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          float bias_raw;
          if constexpr (LIMBS) {
            const int H = butterfly8(hpart, lane);
            const int M = butterfly8(mpart, lane);
            bias_raw = __fadd_rn(__fmul_rn(static_cast<float>(H), 65536.f), static_cast<float>(M));
          } else {
            bias_raw = butterfly8(fpart, lane);
          }
          if (r_out < n) {
            const int64_t v = v0 + r_out;
            // int8: scale_v * 2^-shift * sum; the power of two is applied last so that a
            // tiny embedding row underflows gracefully instead of through 2^-shift.
            float bias = bias_raw;
            if constexpr (INT8) {
              bias = __fmul_rn(bias_raw, scale_v);
              if constexpr (LIMBS) bias = __fmul_rn(__fmul_rn(bias, inv_lo), inv_hi);
            }
            best = umax64(best, score_entry<PROB, LOGITS>(p, b, i, v, base_v, bias, seed, sampled, T_b));
          }
        }
        return best;
      };
      uint64_t best;
      if (INT8 && !float_path) best = row_loop(std::integral_constant<bool, INT8>{});
      else best = row_loop(std::false_type{});

      // CTA argmax for row b. Its W1 row goes towards L2 now: the grid-wide winner is
      // one of the CTAs' local winners, so the next position's embedding load hits L2.
      best = warp_max64(best);
      if (lane == 0) red[warp] = best;
      __syncthreads();
      if (warp == 0) {
        uint64_t x = lane < kWalkWarps ? red[lane] : 0ull;
        x = warp_max64(x);
        if (lane == 0) best_s[b] = x;
        if (x != 0ull && lane < 4 && i + 1 < p.K)
          prefetch_l2(p.w1 + static_cast<size_t>(unpack_idx(x)) * kRank + 64 * lane);
      }
      filled = true;
      __syncthreads();
    }
    for (int t = threadIdx.x; t < p.bs; t += blockDim.x)
      if (prev_s[t] < 0) best_s[t] = 0ull;

    if (!exchange_best(p.sync, i, p.bs, skip0 && i == 0, best_s, flag)) {
      release_tmem();
      return;
    }
    if (i + 2 < p.K) prefetch_base_slice(p, v0, n, i + 2);
    for (int t = threadIdx.x; t < p.bs; t += blockDim.x) {
      const int tok = prev_s[t] >= 0 ? unpack_idx(best_s[t]) : -1;
      prev_s[t] = tok;
      if (cta == 0) p.tokens[static_cast<size_t>(t) * p.K + i] = tok;
    }
    reset_behind(p.sync, i, p.bs);
  }
  release_tmem();
  finish_walk(p.sync, p.K, p.bs, flag);
}

#define DSPARK_INST(I, P, L) template __global__ void walk_cc_kernel<I, P, L>(const WalkParams);
DSPARK_INST(true, false, false)
DSPARK_INST(true, false, true)
DSPARK_INST(true, true, false)
DSPARK_INST(true, true, true)
DSPARK_INST(false, false, false)
DSPARK_INST(false, false, true)
DSPARK_INST(false, true, false)
DSPARK_INST(false, true, true)
#undef DSPARK_INST

// Host-side handle of the kernel variant for (W2 format, mode, draft_logits).
const void* walk_cc_kernel_ptr(bool int8, bool prob, bool logits) {
  if (int8) {
    if (prob) return logits ? (const void*)walk_cc_kernel<true, true, true> : (const void*)walk_cc_kernel<true, true, false>;
    return logits ? (const void*)walk_cc_kernel<true, false, true> : (const void*)walk_cc_kernel<true, false, false>;
  }
  if (prob) return logits ? (const void*)walk_cc_kernel<false, true, true> : (const void*)walk_cc_kernel<false, true, false>;
  return logits ? (const void*)walk_cc_kernel<false, false, true> : (const void*)walk_cc_kernel<false, false, false>;
}

}  // namespace dspark
