// Top-k Markov walk (vLLM PR #49969, "[Spec Decode] Add top-k DSpark Markov
// projection", "Purpose"): the top-k candidates of every draft position are chosen
// once from the base logits, the Markov bias is evaluated for those candidates only
// (their bf16 W2 rows are gathered), and each step's argmax or Gumbel-max sample runs
// over the dense row that is -inf everywhere off the candidates.
//
// topk_select_kernel: one CTA per (b, i) row. Two 256-bin histogram passes over the
// 16-bit orderable key of the bf16 base logits find the k-th largest key T and how
// many entries equal to T are still needed; a third pass compacts, in ascending
// vocabulary order, every entry above T plus the first `need` entries equal to T
// (ties at the boundary go to the smaller index; NaN is the largest key). With
// draft_logits requested it also writes -inf at every non-candidate entry.
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

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;

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

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(const uint16_t* base, int64_t V,
                                                                  int k, int32_t* cand,
                                                                  uint16_t* logits) {
  __shared__ int hist[256];
  __shared__ int scan_sh[80];
  __shared__ int sel[4];
  const size_t row = blockIdx.x;
  const uint16_t* x = base + row * static_cast<size_t>(V);

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
      if (take[t]) cand[row * k + pos++] = static_cast<int32_t>(vb + t);
      else if (logits) logits[row * static_cast<size_t>(V) + vb + t] = 0xFF80u;  // -inf
    }
    eq_seen += eq_total;
    out_base += take_total;
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
  topk_select_kernel<<<rows, kSelThreads, 0, stream>>>(base, V, k, cand, logits);
  return cudaGetLastError();
}

}  // namespace dspark
