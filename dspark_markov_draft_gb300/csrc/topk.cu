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
// over the row collects every entry at or above the pivot into shared memory (warp-
// aggregated appends); T is found by a two-byte radix select on that list; boundary
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


// Per-halfword unsigned maximum of two packed pairs.
__device__ __forceinline__ uint32_t umax_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
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
                                                                  int k, int32_t* cand,
                                                                  uint16_t* logits) {
  extern __shared__ __align__(16) unsigned char sel_smem[];
  int* hist = reinterpret_cast<int*>(sel_smem);                           // [kSelBins]
  uint32_t* lidx = reinterpret_cast<uint32_t*>(hist + kSelBins);           // [kSelCap]
  uint16_t* lkey = reinterpret_cast<uint16_t*>(lidx + kSelCap);            // [kSelCap]
  int* scan_sh = reinterpret_cast<int*>(lkey + kSelCap);                   // [80]
  int* sel = scan_sh + 80;                                                 // [8]
  const int tid = threadIdx.x;
  const size_t row = blockIdx.x;
  const uint16_t* x = base + row * static_cast<size_t>(V);
  int32_t* out = cand + row * static_cast<size_t>(k);

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
        lkey[pos] = static_cast<uint16_t>(key16(x[v]));
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
    uint4 w[4], wn[4];
    load4(0, w);
    for (int64_t c0 = 0; c0 < n8; c0 += 4 * kSelThreads) {
      if (c0 + 4 * kSelThreads < n8) load4(c0 + 4 * kSelThreads, wn);  // next batch in flight
      uint32_t take = 0;  // bit 8 j + e: entry 8 (c0 + j kSelThreads + tid) + e
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t c = c0 + j * kSelThreads + tid;
        const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
        // Quick reject of 8 entries: with the pivot above -0, only non-negative
        // entries (whose key is the pattern with the sign bit set) or NaNs can pass.
        if (quick) {
          const uint32_t m = umax_u16x2(umax_u16x2(ww[0] ^ 0x80008000u, ww[1] ^ 0x80008000u),
                                        umax_u16x2(ww[2] ^ 0x80008000u, ww[3] ^ 0x80008000u));
          const uint32_t a = umax_u16x2(umax_u16x2(ww[0] & 0x7FFF7FFFu, ww[1] & 0x7FFF7FFFu),
                                        umax_u16x2(ww[2] & 0x7FFF7FFFu, ww[3] & 0x7FFF7FFFu));
          const bool any_nan = (a & 0xFFFFu) > 0x7F80u || (a >> 16) > 0x7F80u;
          if (!any_nan && (m & 0xFFFFu) < pivot && (m >> 16) < pivot) continue;
        }
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
        const uint32_t kk = lkey[e];
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
    const uint32_t kk = e < n ? lkey[e] : 0u;
    const bool take = e < n && (kk > T || (kk == T && all_ties));
    const int pos = warp_append(take ? 1 : 0, n_out);
    if (take && pos < k) out[pos] = static_cast<int32_t>(lidx[e]);
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
      if (rank < need_eq && *n_out + rank < k) out[*n_out + rank] = static_cast<int32_t>(me);
    }
  }
}

template <bool PROB, bool LOGITS>
__global__ void __launch_bounds__(kWalkThreads, 1) topk_walk_kernel(const WalkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int G = gridDim.x, cta = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j8 = lane & 7, grp = lane >> 3;
  float* e_s = reinterpret_cast<float*>(smem);                 // [bs][256] fp32
  int* prev_s = reinterpret_cast<int*>(e_s + static_cast<size_t>(p.bs) * kRank);
  uint64_t* best_s = reinterpret_cast<uint64_t*>(prev_s + 64);
  uint64_t* red = best_s + 64;
  int* flag = reinterpret_cast<int*>(red + kWalkWarps);

  const int64_t items = static_cast<int64_t>(p.bs) * p.top_k;
  const int64_t lo = static_cast<int64_t>(cta) * items / G;
  const int64_t hi = static_cast<int64_t>(cta + 1) * items / G;
  const bool skip0 = (p.sync.flags & DSPARK_FLAG_SKIP_ARRIVAL_CTA0) && cta == 0;
  const unsigned char* w2g = reinterpret_cast<const unsigned char*>(p.w2);
  constexpr int kRowBytes = 2 * kRank;

  for (int t = threadIdx.x; t < p.bs; t += blockDim.x) {
    const int32_t tok = p.prev[t];
    const bool ok = tok >= 0 && static_cast<int64_t>(tok) < p.V;
    prev_s[t] = ok ? tok : -1;
    if (!ok && cta == 0) report(p.sync.status_dev, DSPARK_ERR_BAD_TOKEN);
  }

  for (int i = 0; i < p.K; ++i) {
    __syncthreads();
    for (int t = threadIdx.x; t < p.bs; t += blockDim.x) best_s[t] = 0ull;
    for (int b = warp; b < p.bs; b += kWalkWarps) {
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

    const int b_first = lo < hi ? static_cast<int>(lo / p.top_k) : 0;
    const int b_last = lo < hi ? static_cast<int>((hi - 1) / p.top_k) : -1;
    for (int b = b_first; b <= b_last; ++b) {
      if (prev_s[b] < 0) continue;
      const int64_t j_lo = max(lo, static_cast<int64_t>(b) * p.top_k) - static_cast<int64_t>(b) * p.top_k;
      const int64_t j_hi = min(hi, static_cast<int64_t>(b + 1) * p.top_k) - static_cast<int64_t>(b) * p.top_k;
      const int32_t* cand = p.cand + (static_cast<size_t>(b) * p.K + i) * p.top_k;
      const uint64_t seed = PROB ? p.seeds[b] : 0ull;
      float ef[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) ef[c] = e_s[static_cast<size_t>(b) * kRank + (j8 + 8 * (c / 8)) * 8 + (c % 8)];

      uint64_t best = 0ull;
      for (int64_t r0 = j_lo + 32 * warp; r0 < j_hi; r0 += 32 * kWalkWarps) {
        const int64_t rbase = r0 + 8 * grp;
        float part[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int64_t r = rbase + rr;
          float a = 0.f;
          if (r < j_hi) {
            const int64_t cv = min(max(static_cast<int64_t>(cand[r]), int64_t{0}), p.V - 1);
            const unsigned char* row = w2g + static_cast<size_t>(cv) * kRowBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 q = __ldg(reinterpret_cast<const uint4*>(row) + j8 + 8 * c);
              const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                a = __fmaf_rn(bf16_lo(qw[w]), ef[8 * c + 2 * w], a);
                a = __fmaf_rn(bf16_hi(qw[w]), ef[8 * c + 2 * w + 1], a);
              }
            }
          }
          part[rr] = a;
        }
        // butterfly over the 8 lanes of the group (same tree as the dense walk)
        const bool u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float send = u4 ? part[t] : part[t + 4];
          const float keep = u4 ? part[t + 4] : part[t];
          part[t] = keep + __shfl_xor_sync(kFull, send, 4);
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float send = u2 ? part[t] : part[t + 2];
          const float keep = u2 ? part[t + 2] : part[t];
          part[t] = keep + __shfl_xor_sync(kFull, send, 2);
        }
        const float send = u1 ? part[0] : part[1];
        const float keep = u1 ? part[1] : part[0];
        const float bias = keep + __shfl_xor_sync(kFull, send, 1);

        const int64_t r = rbase + j8;
        if (r < j_hi) {
          const int64_t v = min(max(static_cast<int64_t>(cand[r]), int64_t{0}), p.V - 1);
          const size_t o = (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(p.V) + v;
          const float l = __fadd_rn(bf16_to_f32(p.base[o]), bias);
          if (LOGITS) p.logits[o] = f32_to_bf16_bits(l);
          float s = l;
          if (PROB) {
            const float lb = bf16_to_f32(f32_to_bf16_bits(l));
            const float xs = p.temp_is_one ? lb : __fdiv_rn(lb, p.temperature);
            const uint4 w = philox_block(seed, b, i, static_cast<uint32_t>(v >> 2));
            s = __fadd_rn(xs, gumbel_from_word(uint4_get(w, static_cast<int>(v & 3))));
          }
          best = umax64(best, pack_best(order_key(s), static_cast<uint32_t>(v)));
        }
      }
      best = warp_max64(best);
      if (lane == 0) red[warp] = best;
      __syncthreads();
      if (warp == 0) {
        uint64_t xw = lane < kWalkWarps ? red[lane] : 0ull;
        xw = warp_max64(xw);
        if (lane == 0) best_s[b] = umax64(best_s[b], xw);
        if (xw != 0ull && lane < 4 && i + 1 < p.K)
          prefetch_l2(p.w1 + static_cast<size_t>(unpack_idx(xw)) * kRank + 64 * lane);
      }
      __syncthreads();
    }

    if (!exchange_best(p.sync, i, p.bs, skip0 && i == 0, best_s, flag)) return;
    for (int t = threadIdx.x; t < p.bs; t += blockDim.x) {
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

const void* topk_walk_kernel_ptr(bool prob, bool logits) {
  if (prob) return logits ? (const void*)topk_walk_kernel<true, true> : (const void*)topk_walk_kernel<true, false>;
  return logits ? (const void*)topk_walk_kernel<false, true> : (const void*)topk_walk_kernel<false, false>;
}

cudaError_t launch_topk_select(const uint16_t* base, int64_t V, int k, int rows, int32_t* cand,
                               uint16_t* logits, cudaStream_t stream) {
  constexpr size_t smem = kSelBins * 4 + kSelCap * 6 + 96 * 4;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  topk_select_kernel<<<rows, kSelThreads, smem, stream>>>(base, V, k, cand, logits);
  return cudaGetLastError();
}

}  // namespace dspark
