// Top-k Markov walk (vLLM PR #49969, "[Spec Decode] Add top-k DSpark Markov
// projection", "Purpose"): the top-k candidates of every draft position are chosen
// once from the base logits, the Markov bias is evaluated for those candidates only
// (their bf16 W2 rows are gathered), and each step's argmax or Gumbel-max sample runs
// over the dense row that is -inf everywhere off the candidates.
//
// topk_select_kernel: one CTA per (b, i) row; candidates are written in no particular
// order (only the set matters). Keys are 16-bit orderable keys of the bf16 base logits
// (NaN largest, -0 equal to +0); the set is every entry with key above the k-th
// largest key T plus, among the entries equal to T, the ones with the smallest
// vocabulary indices. Fast path: a histogram of the 11-bit key prefix of ~4096 evenly
// spaced samples gives a pivot prefix that at least ~1.15 k entries reach; one pass
// over the row collects every entry at or above the pivot into shared memory (a pivot
// above +0 is tested on two packed entries at once, without branches; warp-aggregated
// appends); T is found by a two-byte radix select on that list; boundary
// ties are resolved by ranking the tied indices. Rows where the pivot collects fewer
// than k or more than kSelCap entries, or the tie at T is wider than kSelTies, take the
// exact path over the whole row: two 256-bin histogram passes and an ordered
// compaction. With draft_logits requested the row is first filled with -inf (the walk
// writes the candidates).
//
// topk_walk_kernel: persistent cooperative kernel over the K positions; the bs*k
// (row, candidate) items are split evenly over the grid; 8 lanes share a gathered W2
// row exactly as in the dense walk, then the same per-step argmax atomics and
// bounded barrier. An all -inf candidate set yields token 0, the dense-row argmax.
#include <cstdint>

#include "common.cuh"
#include "walk_params.cuh"

namespace dspark {

namespace {

// L2 policies of the candidate walk: W2 rows are read again at later positions (evict
// last); candidate ids and their base logits are read once (evict first, no L1 line).
__device__ __forceinline__ uint64_t l2_policy_keep() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_once() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_keep_u4(const void* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ld_once_b32(const void* ptr, uint64_t pol) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ uint32_t ld_once_u16(const uint16_t* ptr, uint64_t pol) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(v) : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void prefetch_l2_keep(const void* ptr) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(ptr));
}

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCap = 8192;    // entries collected by the fast path
constexpr int kSelTies = 2048;   // widest tie at the k-th key the fast path resolves
constexpr int kSelBins = 2048;   // 11-bit key prefixes
constexpr int kSelSamples = 4096;

// Orderable 16-bit key of a bf16 pattern: NaN largest, -0 equal to +0.
__device__ __forceinline__ uint32_t key16(uint16_t h) {
  if ((h & 0x7FFFu) > 0x7F80u) return 0xFFFFu;
  if ((h & 0x7FFFu) == 0u) h = 0;
  return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// Block-wide exclusive scan of one int per thread; returns the prefix and the total.
__device__ __forceinline__ int block_exscan(int x, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelWarps ? sh[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kSelWarps) sh[32 + lane] = wi - w;
    if (lane == kSelWarps - 1) sh[64] = wi;
  }
  __syncthreads();
  const int res = sh[32 + warp] + incl - x;
  total = sh[64];
  __syncthreads();
  return res;
}

}  // namespace

// Exact selection over the whole row (the fast path's fallback): candidates in
// ascending vocabulary order.
__device__ void select_exact(const uint16_t* x, int64_t V, int k, int32_t* out, int* hist,
                             int* scan_sh, int* sel) {

  // Pass 1 and 2: histograms of the high and then the low byte of the key.
  uint32_t prefix = 0;
  int above = 0;  // entries with key strictly above the current bin range
  for (int pass = 0; pass < 2; ++pass) {
    for (int t = threadIdx.x; t < 256; t += blockDim.x) hist[t] = 0;
    __syncthreads();
    for (int64_t v = threadIdx.x; v < V; v += blockDim.x) {
      const uint32_t kk = key16(x[v]);
      if (pass == 0) atomicAdd(&hist[kk >> 8], 1);
      else if ((kk >> 8) == prefix) atomicAdd(&hist[kk & 0xFFu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = above, bin = 0;
      for (int h = 255; h >= 0; --h) {
        if (acc + hist[h] >= k) { bin = h; break; }
        acc += hist[h];
      }
      sel[0] = bin;
      sel[1] = acc;
    }
    __syncthreads();
    prefix = pass == 0 ? static_cast<uint32_t>(sel[0]) : ((prefix << 8) | static_cast<uint32_t>(sel[0]));
    above = sel[1];
    __syncthreads();
  }
  const uint32_t thr = prefix;    // the k-th largest key
  const int need_eq = k - above;  // entries equal to thr still to take (>= 1)

  // Pass 3: ordered compaction, 8 consecutive entries per thread per chunk.
  int eq_seen = 0, out_base = 0;
  const int64_t chunk = static_cast<int64_t>(kSelThreads) * 8;
  for (int64_t c0 = 0; c0 < V; c0 += chunk) {
    const int64_t vb = c0 + static_cast<int64_t>(threadIdx.x) * 8;
    uint32_t keys[8];
    int n_eq = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      keys[t] = (vb + t < V) ? key16(x[vb + t]) : 0u;
      n_eq += (vb + t < V && keys[t] == thr) ? 1 : 0;
    }
    int eq_total;
    int eq_pre = block_exscan(n_eq, scan_sh, eq_total) + eq_seen;
    bool take[8];
    int n_take = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const bool in = vb + t < V;
      bool tk = in && keys[t] > thr;
      if (in && keys[t] == thr) { tk = eq_pre < need_eq; ++eq_pre; }
      take[t] = tk;
      n_take += tk ? 1 : 0;
    }
    int take_total;
    int pos = block_exscan(n_take, scan_sh, take_total) + out_base;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      if (vb + t >= V) continue;
      if (take[t]) out[pos++] = static_cast<int32_t>(vb + t);
    }
    eq_seen += eq_total;
    out_base += take_total;
  }
}



// Warp-aggregated append: every lane adds `c` items; returns this lane's first slot of
// a block-wide counter (all lanes of the warp call it).
__device__ __forceinline__ int warp_append(int c, int* counter) {
  const int lane = threadIdx.x & 31;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  int base = 0;
  if (lane == 31) base = atomicAdd(counter, incl);
  base = __shfl_sync(kFull, base, 31);
  return base + incl - c;
}

__global__ void __launch_bounds__(kSelThreads, 3) topk_select_kernel(const uint16_t* base, int64_t V,
                                                                  int k, int32_t* cand, float* cand_base,
                                                                  uint16_t* logits) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  int* hist = reinterpret_cast<int*>(sel_smem);                           // [kSelBins]
  uint32_t* lidx = reinterpret_cast<uint32_t*>(hist + kSelBins);           // [kSelCap]
  uint16_t* lval = reinterpret_cast<uint16_t*>(lidx + kSelCap);            // [kSelCap] bf16 bits
  int* scan_sh = reinterpret_cast<int*>(lval + kSelCap);                   // [80]
  int* sel = scan_sh + 80;                                                 // [8]
  const int tid = threadIdx.x;
  const size_t row = blockIdx.x;
  const uint16_t* x = base + row * static_cast<size_t>(V);
  int32_t* out = cand + row * static_cast<size_t>(k);
  // the candidates' base logits beside their ids (fp32 of the bf16 bits): the walk then
  // reads them contiguously instead of one scattered entry of the dense row each
  float* out_base = cand_base + row * static_cast<size_t>(k);

  if (logits) {  // -inf everywhere; the walk overwrites the candidates
    uint16_t* lr = logits + row * static_cast<size_t>(V);
    for (int64_t v = tid; v < V; v += kSelThreads) lr[v] = 0xFF80u;
  }

  // 1. pivot prefix from a sample histogram
  for (int t = tid; t < kSelBins; t += kSelThreads) hist[t] = 0;
  if (tid < 8) sel[tid] = 0;
  __syncthreads();
  // samples: kSelSamples / 64 blocks of 64 consecutive entries, evenly spaced (whole
  // cache lines); rows shorter than kSelSamples are taken whole
  const int64_t nblk = kSelSamples / 64;
  const int64_t stride = V > kSelSamples ? V / kSelSamples : 1;  // entries per sample
  const int64_t ns = V > kSelSamples ? kSelSamples : V;
  const int64_t bstep = V > kSelSamples ? V / nblk : 0;
  for (int64_t s0 = 0; s0 < ns; s0 += 8 * kSelThreads) {  // loads first, then the atomics
    uint16_t sv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t sj = s0 + j * kSelThreads + tid;
      const int64_t v = V > kSelSamples ? (sj >> 6) * bstep + (sj & 63) : sj;
      sv[j] = sj < ns ? __ldg(x + v) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (s0 + j * kSelThreads + tid < ns) atomicAdd(&hist[key16(sv[j]) >> 5], 1);
  }
  __syncthreads();
  // bins in descending order, 4 per thread: the largest prefix whose suffix count
  // reaches the target
  const int target = static_cast<int>(static_cast<double>(k) * 1.15 / static_cast<double>(stride)) + 12;
  int c4 = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) c4 += hist[kSelBins - 1 - (4 * tid + t)];
  int total;
  const int before = block_exscan(c4, scan_sh, total);
  if (tid == 0) sel[0] = 0;  // pivot prefix (0: collect everything)
  __syncthreads();
  if (before < target && before + c4 >= target) {
    int acc = before;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int bin = kSelBins - 1 - (4 * tid + t);
      acc += hist[bin];
      if (acc >= target) { sel[0] = bin; break; }
    }
  }
  __syncthreads();
  const uint32_t pivot = static_cast<uint32_t>(sel[0]) << 5;

  // 2. collect every entry with key >= pivot: 16-byte loads of 8 entries, four per
  // thread in flight, when the row is 16-byte aligned; single entries otherwise
  int* n_col = sel + 1;
  auto append = [&](uint32_t take, auto index_of) {
    int pos = warp_append(__popc(take), n_col);
    while (take) {
      const int t = __ffs(take) - 1;
      take &= take - 1;
      const int64_t v = index_of(t);
      if (pos < kSelCap) {
        lidx[pos] = static_cast<uint32_t>(v);
        lval[pos] = x[v];
      }
      ++pos;
    }
  };
  if ((V & 7) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
    const uint4* x4 = reinterpret_cast<const uint4*>(x);
    const int64_t n8 = V / 8;
    auto load4 = [&](int64_t c0, uint4 (&w)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t c = c0 + j * kSelThreads + tid;
        w[j] = c < n8 ? __ldg(x4 + c) : make_uint4(0, 0, 0, 0);
      }
    };
    const bool quick = pivot > 0x8000u;  // pivot above the keys of -0 / +0
    // With the pivot above +0 an entry passes iff it is a NaN or non-negative with
    // pattern >= pv = pivot - 0x8000 (its key is the pattern with the sign bit set).
    // Both tests on two 16-bit entries at once without carries between the halves:
    // for a magnitude y < 0x8000, y + (0x8000 - pv) has bit 15 set iff y >= pv, and
    // y + 0x7F has it iff y > 0x7F80 (NaN).
    const uint32_t pv = pivot - 0x8000u;
    const uint32_t d2 = (0x8000u - pv) * 0x00010001u;
    uint4 w[4], wn[4];
    load4(0, w);
    for (int64_t c0 = 0; c0 < n8; c0 += 4 * kSelThreads) {
      if (c0 + 4 * kSelThreads < n8) load4(c0 + 4 * kSelThreads, wn);  // next batch in flight
      if (quick) {
        // bit 4 j + jj (+16 for the high half): entry 8 (c0 + j kSelThreads + tid) + 2 jj (+1);
        // the zero words past the row never pass
        uint32_t take = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t y = ww[jj] & 0x7FFF7FFFu;
            const uint32_t r = (((y + d2) & ~ww[jj]) | (y + 0x007F007Fu)) & 0x80008000u;
            take |= r >> (15 - (4 * j + jj));
          }
        }
        append(take, [&](int t) {
          const int hi = t >> 4, j = (t >> 2) & 3, jj = t & 3;
          return 8 * (c0 + j * kSelThreads + tid) + 2 * jj + hi;
        });
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = wn[j];
        continue;
      }
      uint32_t take = 0;  // bit 8 j + e: entry 8 (c0 + j kSelThreads + tid) + e
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t c = c0 + j * kSelThreads + tid;
        const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint16_t h = static_cast<uint16_t>((e & 1) ? (ww[e >> 1] >> 16) : (ww[e >> 1] & 0xFFFFu));
          if (c < n8 && key16(h) >= pivot) take |= 1u << (8 * j + e);
        }
      }
      append(take, [&](int t) { return 8 * (c0 + (t >> 3) * kSelThreads + tid) + (t & 7); });
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = wn[j];
    }
  } else {
    for (int64_t v0 = 0; v0 < V; v0 += 32 * kSelThreads) {
      uint32_t take = 0;  // bit t: entry v0 + t kSelThreads + tid
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int64_t v = v0 + static_cast<int64_t>(t) * kSelThreads + tid;
        if (v < V && key16(x[v]) >= pivot) take |= 1u << t;
      }
      append(take, [&](int t) { return v0 + static_cast<int64_t>(t) * kSelThreads + tid; });
    }
  }
  __syncthreads();
  const int n = *n_col;
  bool exact = n < k || n > kSelCap;

  // 3. k-th largest key T on the list (two byte passes)
  uint32_t T = 0;
  int above = 0, n_eq = 0;
  if (!exact) {
    uint32_t prefix = 0;
    for (int pass = 0; pass < 2; ++pass) {
      for (int t = tid; t < 256; t += kSelThreads) hist[t] = 0;
      __syncthreads();
      for (int e = tid; e < n; e += kSelThreads) {
        const uint32_t kk = key16(lval[e]);
        if (pass == 0) atomicAdd(&hist[kk >> 8], 1);
        else if ((kk >> 8) == prefix) atomicAdd(&hist[kk & 0xFFu], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int acc = above, bin = 0;
        for (int h = 255; h >= 0; --h) {
          if (acc + hist[h] >= k) { bin = h; break; }
          acc += hist[h];
        }
        sel[2] = bin;
        sel[3] = acc;
        sel[4] = hist[bin];
      }
      __syncthreads();
      prefix = pass == 0 ? static_cast<uint32_t>(sel[2]) : ((prefix << 8) | static_cast<uint32_t>(sel[2]));
      above = sel[3];
      n_eq = sel[4];
      __syncthreads();
    }
    T = prefix;
    if (n_eq > k - above && n_eq > kSelTies) exact = true;
  }
  if (exact) {
    select_exact(x, V, k, out, hist, scan_sh, sel);
    __syncthreads();  // the block's ids are written
    for (int j = tid; j < k; j += kSelThreads) out_base[j] = bf16_to_f32(x[out[j]]);
    return;
  }
  const int need_eq = k - above;  // 1 <= need_eq <= n_eq

  // 4. output: every key above T, and the need_eq smallest indices among keys == T
  int* n_out = sel + 5;
  int* n_tie = sel + 6;
  if (tid == 0) { *n_out = 0; *n_tie = 0; }
  __syncthreads();
  uint32_t* ties = reinterpret_cast<uint32_t*>(hist);  // reused: [kSelTies]
  const bool all_ties = need_eq == n_eq;
  for (int e0 = 0; e0 < n; e0 += kSelThreads) {
    const int e = e0 + tid;
    const uint32_t kk = e < n ? key16(lval[e]) : 0u;
    const bool take = e < n && (kk > T || (kk == T && all_ties));
    const int pos = warp_append(take ? 1 : 0, n_out);
    if (take && pos < k) {
      out[pos] = static_cast<int32_t>(lidx[e]);
      out_base[pos] = bf16_to_f32(lval[e]);
    }
    if (!all_ties) {
      const bool tie = e < n && kk == T;
      const int tp = warp_append(tie ? 1 : 0, n_tie);
      if (tie) ties[tp] = lidx[e];
    }
  }
  __syncthreads();
  if (!all_ties) {
    for (int e = tid; e < n_eq; e += kSelThreads) {
      const uint32_t me = ties[e];
      int rank = 0;
      for (int f = 0; f < n_eq; ++f) rank += ties[f] < me ? 1 : 0;
      if (rank < need_eq && *n_out + rank < k) {
        out[*n_out + rank] = static_cast<int32_t>(me);
        out_base[*n_out + rank] = bf16_to_f32(x[me]);
      }
    }
  }
}

constexpr int kChunk = 2048;  // candidates per chunk of a CTA (its whole range at the configs)

// INT8: the candidates' W2 rows are int8 codes (256 bytes) times the row scale, else
// bf16 rows (512 bytes).
template <bool INT8, bool PROB, bool LOGITS>
__global__ void __launch_bounds__(kWalkThreads, 1) topk_walk_kernel(const WalkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j8 = lane & 7, grp = tid >> 3;                     // 64 groups of 8 lanes
  constexpr int kGroups = kWalkThreads / 8;
  float* e_s = reinterpret_cast<float*>(smem);                 // [bs][256] fp32
  int32_t* it_v = reinterpret_cast<int32_t*>(e_s + static_cast<size_t>(p.bs) * kRank);  // [kChunk]
  float* it_base = reinterpret_cast<float*>(it_v + kChunk);    // [kChunk] base logit
  float* it_g = it_base + kChunk;                              // [kChunk] Gumbel noise
  int* prev_s = reinterpret_cast<int*>(it_g + kChunk);         // [64]
  uint64_t* best_s = reinterpret_cast<uint64_t*>(prev_s + 64); // [64]
  int* flag = reinterpret_cast<int*>(best_s + 64);

  // This CTA's candidates: a contiguous range of the bs * k (row, candidate) items,
  // walked in chunks of at most kChunk items.
  const int64_t items = static_cast<int64_t>(p.bs) * p.top_k;
  const int64_t lo = static_cast<int64_t>(cta) * items / G;
  const int64_t hi = static_cast<int64_t>(cta + 1) * items / G;
  const bool skip0 = (p.sync.flags & DSPARK_FLAG_SKIP_ARRIVAL_CTA0) && cta == 0;
  const unsigned char* w2g = INT8 ? reinterpret_cast<const unsigned char*>(p.w2q)
                                  : reinterpret_cast<const unsigned char*>(p.w2);
  constexpr int kRowBytes = INT8 ? kRank : 2 * kRank;
  constexpr int kLaneChunks = kRowBytes / 16 / 8;  // 16-byte chunks j8 + 8 c of a row per lane
  const uint64_t keep = l2_policy_keep(), once = l2_policy_once();

  for (int t = tid; t < p.bs; t += blockDim.x) {
    const int32_t tok = p.prev[t];
    const bool ok = tok >= 0 && static_cast<int64_t>(tok) < p.V;
    const bool settings = row_settings_ok(p, PROB, t);
    prev_s[t] = ok && settings ? tok : -1;
    if (!ok && cta == 0) report(p.sync.status_dev, DSPARK_ERR_BAD_TOKEN);
    if (!settings && cta == 0) report(p.sync.status_dev, DSPARK_ERR_INVALID_ARG);
  }

  // Phase P of position i for the chunk [c_lo, c_hi): everything that does not depend on
  // the previous token -- candidate id, base logit, Gumbel noise -- and the W2 row
  // towards L2.
  auto phase_p = [&](int i, int64_t c_lo, int64_t c_hi) {
    for (int64_t it = c_lo + tid; it < c_hi; it += blockDim.x) {
      const int e = static_cast<int>(it - c_lo);
      const int b = static_cast<int>(it / p.top_k);
      const int64_t j = it - static_cast<int64_t>(b) * p.top_k;
      const size_t ci = (static_cast<size_t>(b) * p.K + i) * p.top_k + j;
      const int64_t v = min(max(static_cast<int64_t>(static_cast<int32_t>(ld_once_b32(p.cand + ci, once))),
                                int64_t{0}), p.V - 1);
      it_v[e] = static_cast<int32_t>(v);
      it_base[e] = p.cand_base
                       ? __uint_as_float(ld_once_b32(p.cand_base + ci, once))
                       : bf16_to_f32(static_cast<uint16_t>(
                             ld_once_u16(p.base + (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v, once)));
      float g = 0.f;
      if (row_sampled(p, PROB, b)) {
        const uint4 w = philox_block(p.seeds[b], b, i, static_cast<uint32_t>(v >> 2));
        g = gumbel_from_word(uint4_get(w, static_cast<int>(v & 3)));
      }
      it_g[e] = g;
      const unsigned char* row = w2g + static_cast<size_t>(v) * kRowBytes;
#pragma unroll
      for (int m = 0; m < kRowBytes / 128; ++m) prefetch_l2_keep(row + 128 * m);
    }
  };

  bool have_p = false;  // phase P of the first chunk of position i already done
  if (lo < hi) {
    phase_p(0, lo, min(hi, lo + kChunk));
    have_p = true;
  }

  for (int i = 0; i < p.K; ++i) {
    __syncthreads();
    for (int t = tid; t < p.bs; t += blockDim.x) best_s[t] = 0ull;
    // embeddings of the rows this CTA touches, as fp32
    const int b_first = lo < hi ? static_cast<int>(lo / p.top_k) : 0;
    const int b_last = lo < hi ? static_cast<int>((hi - 1) / p.top_k) : -1;
    for (int b = b_first + warp; b <= b_last; b += kWalkWarps) {
      const int tok = prev_s[b];
      if (tok < 0) continue;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(tok) * kRank) + lane);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
      float* dst = e_s + static_cast<size_t>(b) * kRank + 8 * lane;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        dst[2 * t] = bf16_lo(ww[t]);
        dst[2 * t + 1] = bf16_hi(ww[t]);
      }
    }
    __syncthreads();

    // Phase D: tasks of up to 8 consecutive candidates of one request row; group g of
    // 8 lanes takes tasks g, g + 64, ...; each lane holds 32 of the 256 positions.
    for (int64_t c_lo = lo; c_lo < hi; c_lo += kChunk) {
      const int64_t c_hi = min(hi, c_lo + kChunk);
      if (!have_p) {
        phase_p(i, c_lo, c_hi);
        __syncthreads();
      }
      have_p = false;
      // tasks: the chunk split at row boundaries into runs of 8
      const int b0 = static_cast<int>(c_lo / p.top_k);
      const int64_t first_end = min(c_hi, static_cast<int64_t>(b0 + 1) * p.top_k);  // end of the first row's run
      const int n0 = static_cast<int>(first_end - c_lo);
      const int t0 = (n0 + 7) / 8;                                          // tasks of the first row
      const int ntask = t0 + static_cast<int>((c_hi - first_end + 7) / 8 +
                                              (c_hi - first_end) / p.top_k + 1);  // upper bound
      int cur_b = -1;
      float ef[32];
      bool samp_b = false;  // row cur_b's sampling settings
      float T_b = 1.0f;
      for (int task = grp; task < ntask; task += kGroups) {
        // task -> [e0, e1) in chunk numbering, all in row b
        int64_t s0;
        int b;
        int64_t e_end;
        if (task < t0) {
          s0 = c_lo + 8 * task;
          b = b0;
          e_end = first_end;
        } else {
          // later rows start at first_end; each row has k candidates (the last may be cut)
          const int64_t kk = p.top_k;
          const int64_t tasks_per_row = (kk + 7) / 8;
          const int64_t rt = task - t0;
          const int64_t rrow = rt / tasks_per_row;
          const int64_t rstart = first_end + rrow * kk;
          s0 = rstart + 8 * (rt - rrow * tasks_per_row);
          b = b0 + 1 + static_cast<int>(rrow);
          e_end = min(c_hi, rstart + kk);
        }
        if (s0 >= e_end) continue;  // past the chunk (uniform per group)
        if (prev_s[b] < 0) continue;
        const int e0 = static_cast<int>(s0 - c_lo);
        const int nt = static_cast<int>(e_end - s0 < 8 ? e_end - s0 : 8);
        if (b != cur_b) {
          // the lane's 32 embedding values: positions 16 (j8 + 8 c) .. + 15 (int8 chunks
          // of 16 codes) or 8 (j8 + 8 c) .. + 7 (bf16 chunks of 8 values)
          constexpr int kPer = 32 / kLaneChunks;  // values per chunk
#pragma unroll
          for (int c = 0; c < kLaneChunks; ++c)
#pragma unroll
            for (int f = 0; f < kPer / 4; ++f) {
              const float4 x4 = *reinterpret_cast<const float4*>(e_s + static_cast<size_t>(b) * kRank +
                                                                 (j8 + 8 * c) * kPer + 4 * f);
              ef[kPer * c + 4 * f + 0] = x4.x; ef[kPer * c + 4 * f + 1] = x4.y;
              ef[kPer * c + 4 * f + 2] = x4.z; ef[kPer * c + 4 * f + 3] = x4.w;
            }
          samp_b = row_sampled(p, PROB, b);
          T_b = samp_b ? row_temperature(p, b) : 1.0f;
          cur_b = b;
        }
        float part[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two batches of 4 rows: 16 loads in flight per lane
          uint4 q[4][kLaneChunks];
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int r = 4 * h + rr;
            const unsigned char* row = w2g + static_cast<size_t>(it_v[e0 + min(r, nt - 1)]) * kRowBytes;
#pragma unroll
            for (int c = 0; c < kLaneChunks; ++c)
              q[rr][c] = r < nt ? ld_keep_u4(reinterpret_cast<const uint4*>(row) + j8 + 8 * c, keep) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            float a = 0.f;
#pragma unroll
            for (int c = 0; c < kLaneChunks; ++c) {
              const uint32_t qw[4] = {q[rr][c].x, q[rr][c].y, q[rr][c].z, q[rr][c].w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                if constexpr (INT8) {
                  // 4 codes, each exact in fp32 (the row scale comes later): the biased
                  // byte q + 128 as the mantissa of 2^23 + q + 128, minus 2^23 + 128
                  const uint32_t bw = qw[w] ^ 0x80808080u;
#pragma unroll
                  for (int e8 = 0; e8 < 4; ++e8) {
                    const float f = __fsub_rn(__uint_as_float(__byte_perm(bw, 0x4B000000u, 0x7650u + e8)), 8388736.0f);
                    a = __fmaf_rn(f, ef[16 * c + 4 * w + e8], a);
                  }
                } else {
                  a = __fmaf_rn(bf16_lo(qw[w]), ef[8 * c + 2 * w], a);
                  a = __fmaf_rn(bf16_hi(qw[w]), ef[8 * c + 2 * w + 1], a);
                }
              }
            }
            part[4 * h + rr] = a;
          }
        }
        // butterfly over the 8 lanes of the group: lane j8 ends with candidate e0 + j8
        const unsigned gmask = 0xFFu << (lane & 24);
        const bool u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float send = u4 ? part[t] : part[t + 4];
          const float keep = u4 ? part[t + 4] : part[t];
          part[t] = keep + __shfl_xor_sync(gmask, send, 4);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float send = u2 ? part[t] : part[t + 2];
          const float keep = u2 ? part[t + 2] : part[t];
          part[t] = keep + __shfl_xor_sync(gmask, send, 2);
        }
        const float send = u1 ? part[0] : part[1];
        const float keep = u1 ? part[1] : part[0];
        float bias = keep + __shfl_xor_sync(gmask, send, 1);

        if (j8 < nt) {
          const int e = e0 + j8;
          const int64_t v = it_v[e];
          if constexpr (INT8) bias = __fmul_rn(bias, __ldg(p.scales + v));
          const float l = __fadd_rn(it_base[e], bias);
          const uint16_t lh = f32_to_bf16_bits(l);
          if (LOGITS) p.logits[(static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v] = lh;
          float sco = l;
          if (samp_b) {
            const float lb = bf16_to_f32(lh);
            const float xs = T_b == 1.0f ? lb : __fdiv_rn(lb, T_b);
            sco = __fadd_rn(xs, it_g[e]);
          }
          atomicMax(reinterpret_cast<unsigned long long*>(&best_s[b]),
                    static_cast<unsigned long long>(pack_best(order_key(sco), static_cast<uint32_t>(v))));
        }
      }
      __syncthreads();  // the chunk's item arrays are free again
    }

    // Prefetch the CTA winners' embedding rows, publish, do the next position's first
    // phase P while the grid arrives, then read the winners back.
    if (tid < p.bs && best_s[tid] != 0ull && i + 1 < p.K) {
      const uint16_t* row = p.w1 + static_cast<size_t>(unpack_idx(best_s[tid])) * kRank;
#pragma unroll
      for (int l4 = 0; l4 < 4; ++l4) prefetch_l2(row + 64 * l4);
    }
    exchange_arrive(p.sync, i, p.bs, skip0 && i == 0, best_s);
    if (i + 1 < p.K && lo < hi) {
      phase_p(i + 1, lo, min(hi, lo + kChunk));
      have_p = true;
    }
    if (!exchange_wait(p.sync, i, p.bs, best_s, flag)) return;
    for (int t = tid; t < p.bs; t += blockDim.x) {
      int tok = -1;
      if (prev_s[t] >= 0) {
        const uint64_t w = best_s[t];
        // Every candidate at -inf: the dense row is -inf everywhere and its argmax is 0.
        tok = (static_cast<uint32_t>(w >> 32) == order_key(__int_as_float(0xFF800000))) ? 0 : unpack_idx(w);
      }
      prev_s[t] = tok;
      if (cta == 0) p.tokens[static_cast<size_t>(t) * p.K + i] = tok;
    }
    reset_behind(p.sync, i, p.bs);
  }
  finish_walk(p.sync, p.K, p.bs, flag);
}

size_t topk_walk_smem(int bs) {
  return static_cast<size_t>(bs) * kRank * 4 + 3 * kChunk * 4 + 64 * 4 + 64 * 8 + 16 + 128;
}

const void* topk_walk_kernel_ptr(bool int8, bool prob, bool logits) {
#define DSPARK_TK(I, P, L) \
  if (int8 == I && prob == P && logits == L) return (const void*)topk_walk_kernel<I, P, L>;
  DSPARK_TK(true, true, true)
  DSPARK_TK(true, true, false)
  DSPARK_TK(true, false, true)
  DSPARK_TK(true, false, false)
  DSPARK_TK(false, true, true)
  DSPARK_TK(false, true, false)
  DSPARK_TK(false, false, true)
  DSPARK_TK(false, false, false)
#undef DSPARK_TK
  return nullptr;
}

cudaError_t launch_topk_select(const uint16_t* base, int64_t V, int k, int rows, int32_t* cand,
                               float* cand_base, uint16_t* logits, cudaStream_t stream) {
  constexpr size_t smem = kSelBins * 4 + kSelCap * 6 + 96 * 4;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  topk_select_kernel<<<rows, kSelThreads, smem, stream>>>(base, V, k, cand, cand_base, logits);
  return cudaGetLastError();
}

}  // namespace dspark
