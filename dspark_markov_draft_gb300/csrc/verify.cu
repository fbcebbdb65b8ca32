// Speculative-sampling verification of the drafted tokens (Leviathan, Kalman, Matias,
// "Fast Inference from Transformers via Speculative Decoding", ICML 2023, Algorithm 1),
// consuming the bf16 draft_logits the walk kept: they are the distribution the draft
// tokens were sampled from (vLLM PR #62958, "Details").
//
// With q_i = softmax(draft[b, i, :] / T) and p_i = softmax(target[b, i, :] / T):
//   for i = 0 .. K-1: accept d_i iff u_i q_i(d_i) < p_i(d_i) (u_i uniform, Philox
//   counter domain 1); at the first rejection emit a sample of norm(max(0, p_i - q_i))
//   and stop; if every draft is accepted, emit a sample of p_K.
// Samples are Gumbel-max draws (counter domain 2): residual scores log(p - q) + g where
// p > q (p > q nowhere: the scores of p), bonus scores target / T + g.
//
// verify_accept_kernel: one CTA per (draft position i, row b): the softmax normalisers
// of the two rows (one pass, running maximum) and the acceptance bit of d_i (atomicOr
// into the row's word).
// verify_emit_kernel: a cluster of kEmitCtas CTAs per row, each on a vocabulary slice
// (launched as a programmatic dependent of the acceptance kernel, which it waits for):
// the accepted prefix from the bits, then the sample at the first rejected position
// (or the bonus) -- only there -- with the slices' partial normalisers and argmax words
// exchanged through distributed shared memory; rank 0 writes the emitted sequence.
#include <cstdint>

#include <cooperative_groups.h>

#include "common.cuh"

namespace dspark {

namespace {

namespace cg = cooperative_groups;

constexpr int kVerifyThreads = 256;
constexpr int kVerifyWarps = kVerifyThreads / 32;
constexpr int kEmitCtas = 8;
constexpr float kLog2e = 1.4426950408889634f;

// The drafter's Philox4x32-10 generator in another counter domain (the last counter
// word, 0 for the drafter): 1 for the acceptance uniforms, 2 for the resampling noise.
__device__ __forceinline__ uint4 philox_block_d(uint64_t seed, int b, int i, uint32_t m, uint32_t domain) {
  return philox4x32_10(make_uint4(m, static_cast<uint32_t>(i), static_cast<uint32_t>(b), domain),
                       static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

// Hardware base-2 exponential (relative error about 2^-22; 2^-inf = 0; results below
// 2^-126 flush to 0, which no normaliser or acceptance test here can notice).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Hardware reciprocal (about 1 ulp); used on arguments in [6e-8, 17].
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct VerifyParams {
  const uint16_t* target;   // [bs, K+1, V]
  const uint16_t* draft;    // [bs, K, V]
  const int32_t* dtok;      // [bs, K]
  const uint64_t* seeds;    // [bs]
  int64_t V;
  int32_t bs, K;
  float inv_t;              // 1 / T rounded to fp32
  int32_t* accepted;        // [bs]: acceptance bits, then the accepted count
  int32_t* out_tokens;      // [bs, K+1]
  float4* norms;            // [bs, K]: (target max, target sum, draft max, draft sum), or null
};

// Softmax of row / T as a running maximum m of the raw values and z = sum 2^((x - m) c),
// c = log2(e) / T. The probability of x is 2^((x - m) c) / z (0 for an all -inf row).
struct Softmax {
  float m, z;
};

// One entry into a running softmax (the path for unaligned rows).
__device__ __forceinline__ void sm_add(Softmax& s, float x, float c) {
  if (x > s.m) {
    s.z = s.m > -INFINITY ? __fadd_rn(__fmul_rn(s.z, ex2(__fmul_rn(__fsub_rn(s.m, x), c))), 1.f) : 1.f;
    s.m = x;
  } else if (x > -INFINITY) {
    s.z = __fadd_rn(s.z, ex2(__fmul_rn(__fsub_rn(x, s.m), c)));
  }
}

// A chunk of kChunk entries into a running softmax: the chunk maximum first, one
// rescale of z if it rises, then one exponential per entry, 2^(x c - m c) (a fused
// multiply-add; x = -inf gives 0).
template <int kChunk>
__device__ __forceinline__ void sm_add_chunk(Softmax& s, const float (&x)[kChunk], float c) {
  float cm = x[0];
#pragma unroll
  for (int k = 1; k < kChunk; ++k) cm = fmaxf(cm, x[k]);
  if (cm > s.m) {
    s.z = s.m > -INFINITY ? __fmul_rn(s.z, ex2(__fmul_rn(__fsub_rn(s.m, cm), c))) : 0.f;
    s.m = cm;
  }
  if (s.m > -INFINITY) {
    const float nmc = -__fmul_rn(s.m, c);
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int k = 0; k < kChunk; k += 2) {
      z0 = __fadd_rn(z0, ex2(__fmaf_rn(x[k], c, nmc)));
      z1 = __fadd_rn(z1, ex2(__fmaf_rn(x[k + 1], c, nmc)));
    }
    s.z = __fadd_rn(s.z, __fadd_rn(z0, z1));
  }
}

__device__ __forceinline__ Softmax sm_combine(Softmax a, Softmax b, float c) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f};
  const float za = a.m > -INFINITY ? __fmul_rn(a.z, ex2(__fmul_rn(__fsub_rn(a.m, m), c))) : 0.f;
  const float zb = b.m > -INFINITY ? __fmul_rn(b.z, ex2(__fmul_rn(__fsub_rn(b.m, m), c))) : 0.f;
  return {m, __fadd_rn(za, zb)};
}

__device__ __forceinline__ Softmax sm_reduce_cta(Softmax s, float c, Softmax* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    s = sm_combine(s, Softmax{__shfl_xor_sync(kFull, s.m, o), __shfl_xor_sync(kFull, s.z, o)}, c);
  __syncthreads();  // sh free again
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
  __syncthreads();
  s = sh[0];
  for (int w = 1; w < kVerifyWarps; ++w) s = sm_combine(s, sh[w], c);
  return s;
}

// The normalisers of ta[v0, v1) and tb[v0, v1) (two bf16 rows), reduced over the CTA:
// kUnroll 16-byte loads per row in flight per thread when both rows are 16-byte aligned
// and V, v0 are multiples of 8, else single entries.
template <int kUnroll>
__device__ void softmax_pair(const uint16_t* ta, const uint16_t* tb, int64_t V, int64_t v0, int64_t v1,
                             float c, Softmax* sh, Softmax& sa, Softmax& sb) {
  Softmax a{-INFINITY, 0.f}, b{-INFINITY, 0.f};
  const int tid = threadIdx.x;
  if ((V & 7) == 0 && (v0 & 7) == 0 &&
      ((reinterpret_cast<uintptr_t>(ta) | reinterpret_cast<uintptr_t>(tb)) & 15u) == 0) {
    const uint4* a4 = reinterpret_cast<const uint4*>(ta);
    const uint4* b4 = reinterpret_cast<const uint4*>(tb);
    const int64_t c1 = v1 / 8;
    const uint4 ninf = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // bf16 -inf
    for (int64_t c0 = v0 / 8; c0 < c1; c0 += kUnroll * kVerifyThreads) {
      uint4 wa[kUnroll], wb[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t q = c0 + u * kVerifyThreads + tid;
        wa[u] = q < c1 ? __ldg(a4 + q) : ninf;
        wb[u] = q < c1 ? __ldg(b4 + q) : ninf;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const uint32_t ua[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
        const uint32_t ub[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
        float xa[8], xb[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          xa[2 * k] = bf16_lo(ua[k]);
          xa[2 * k + 1] = bf16_hi(ua[k]);
          xb[2 * k] = bf16_lo(ub[k]);
          xb[2 * k + 1] = bf16_hi(ub[k]);
        }
        sm_add_chunk(a, xa, c);
        sm_add_chunk(b, xb, c);
      }
    }
  } else {
    for (int64_t v = v0 + tid; v < v1; v += kVerifyThreads) {
      sm_add(a, bf16_to_f32(__ldg(ta + v)), c);
      sm_add(b, bf16_to_f32(__ldg(tb + v)), c);
    }
  }
  sa = sm_reduce_cta(a, c, sh);
  sb = sm_reduce_cta(b, c, sh);
}

template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T x, Op op, T* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = op(x, __shfl_xor_sync(kFull, x, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = x;
  __syncthreads();
  x = sh[0];
  for (int w = 1; w < kVerifyWarps; ++w) x = op(x, sh[w]);
  return x;
}

__global__ void __launch_bounds__(kVerifyThreads, 4) verify_accept_kernel(const VerifyParams p) {
  __shared__ Softmax sh[kVerifyWarps];
  const int i = blockIdx.x, b = blockIdx.y;
  const int64_t V = p.V;
  const float c = __fmul_rn(kLog2e, p.inv_t);
  const uint16_t* trow = p.target + (static_cast<size_t>(b) * (p.K + 1) + i) * static_cast<size_t>(V);
  const uint16_t* drow = p.draft + (static_cast<size_t>(b) * p.K + i) * static_cast<size_t>(V);
  Softmax st, sd;
  softmax_pair<4>(trow, drow, V, 0, V, c, sh, st, sd);
  // the normalisers of both rows, for the sample pass at this row's emitting position
  if (p.norms && threadIdx.x == 0) p.norms[static_cast<size_t>(b) * p.K + i] = make_float4(st.m, st.z, sd.m, sd.z);
  if (threadIdx.x == 0) {
    const int32_t d = p.dtok[static_cast<size_t>(b) * p.K + i];
    const bool in = d >= 0 && static_cast<int64_t>(d) < V;
    auto prob = [&](const Softmax& s, float x) {
      return s.z > 0.f ? __fdiv_rn(ex2(__fmul_rn(__fsub_rn(x, s.m), c)), s.z) : 0.f;
    };
    const float pd = in ? prob(st, bf16_to_f32(trow[d])) : 0.f;
    const float qd = in ? prob(sd, bf16_to_f32(drow[d])) : 0.f;
    const uint32_t w = philox_block_d(p.seeds[b], b, i, 0u, 1u).x;
    const float u = __fmul_rn(static_cast<float>(2u * (w >> 9) + 1u), 0x1p-24f);  // exact
    if (__fmul_rn(u, qd) < pd) atomicOr(reinterpret_cast<unsigned*>(p.accepted + b), 1u << i);
  }
}

// Start of the vocabulary slice of cluster rank r: a multiple of 8, so that groups of
// four noise words and 16-byte loads stay inside one slice.
__device__ __forceinline__ int64_t emit_slice(int r, int64_t V) {
  return r >= kEmitCtas ? V : (static_cast<int64_t>(r) * V / kEmitCtas) & ~static_cast<int64_t>(7);
}

__global__ void __cluster_dims__(kEmitCtas, 1, 1) __launch_bounds__(kVerifyThreads, 4)
    verify_emit_kernel(const VerifyParams p) {
  __shared__ Softmax sh[kVerifyWarps];
  __shared__ uint64_t shu[kVerifyWarps];
  __shared__ int shi[kVerifyWarps];
  __shared__ Softmax part_t, part_d;  // this slice's normalisers
  __shared__ uint64_t part_best[2];   // this slice's argmax word, per sampling round
  __shared__ int part_any;            // this slice holds an entry with p > q
  wait_previous_kernel();  // the acceptance bits (launched as the acceptance pass's dependent)
  cg::cluster_group cl = cg::this_cluster();
  const int r = static_cast<int>(cl.block_rank()), b = blockIdx.y, tid = threadIdx.x;
  const int64_t V = p.V, v0 = emit_slice(r, V), v1 = emit_slice(r + 1, V);
  const float c = __fmul_rn(kLog2e, p.inv_t);
  // read before the first cluster barrier: rank 0 overwrites it after the second
  const uint32_t bits = static_cast<uint32_t>(p.accepted[b]);
  int n = 0;
  while (n < p.K && ((bits >> n) & 1u)) ++n;
  const uint64_t seed = p.seeds[b];
  const uint16_t* trow = p.target + (static_cast<size_t>(b) * (p.K + 1) + n) * static_cast<size_t>(V);
  const bool residual = n < p.K;
  const uint16_t* drow = residual ? p.draft + (static_cast<size_t>(b) * p.K + n) * static_cast<size_t>(V) : nullptr;
  // p(x) = 2^((x - mt) c) zt, q(x) = 2^((x - md) c) zd (mt, md = 0 and zt, zd = 0 for
  // an all -inf row, so that its probabilities are 0 and not NaN)
  float mt = 0.f, zt = 0.f, md = 0.f, zd = 0.f;
  if (residual) {
    Softmax st{-INFINITY, 0.f}, sd{-INFINITY, 0.f};
    if (p.norms) {
      // the acceptance pass's normalisers of this position's two rows (uniform over the
      // cluster, so every CTA skips the same cluster barrier)
      const float4 nv = p.norms[static_cast<size_t>(b) * p.K + n];
      st = Softmax{nv.x, nv.y};
      sd = Softmax{nv.z, nv.w};
    } else {
      Softmax pt, pd;
      softmax_pair<2>(trow, drow, V, v0, v1, c, sh, pt, pd);
      if (tid == 0) { part_t = pt; part_d = pd; }
      cl.sync();
      for (int q = 0; q < kEmitCtas; ++q) {  // every CTA combines in the same order
        st = sm_combine(st, *cl.map_shared_rank(&part_t, q), c);
        sd = sm_combine(sd, *cl.map_shared_rank(&part_d, q), c);
      }
    }
    if (st.z > 0.f) { mt = st.m; zt = __frcp_rn(st.z); }
    if (sd.z > 0.f) { md = sd.m; zd = __frcp_rn(sd.z); }
  }
  const float nmt = -__fmul_rn(mt, c), nmd = -__fmul_rn(md, c);
  // Gumbel-max. Residual: the argmax of log(p - q) + g over p > q, taken as the argmax
  // of (p - q) / E with E = -log(u) (g = -log(E)); else the scores of p, x / T + g
  // (bonus position, or p > q nowhere after rounding).
  auto sample = [&](bool res, int round) {
    uint64_t best = 0ull;
    int any = 0;
    // 8-byte loads of a group's four entries when both rows allow them (V a multiple of
    // 4 makes every group of the slice whole); indices fit 32 bits (V < 2^31)
    const bool vec = (V & 3) == 0 &&
                     ((reinterpret_cast<uintptr_t>(trow) | (res ? reinterpret_cast<uintptr_t>(drow) : 0u)) & 7u) == 0;
    const uint32_t e1 = static_cast<uint32_t>(v1);
    for (uint32_t m = static_cast<uint32_t>(v0) / 4 + tid; 4 * m < e1; m += kVerifyThreads) {
      const uint4 w4 = philox_block_d(seed, b, n, m, 2u);
      const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
      float xt[4], xd[4] = {0.f, 0.f, 0.f, 0.f};
      if (vec) {
        const uint2 a = __ldg(reinterpret_cast<const uint2*>(trow) + m);
        xt[0] = bf16_lo(a.x); xt[1] = bf16_hi(a.x); xt[2] = bf16_lo(a.y); xt[3] = bf16_hi(a.y);
        if (res) {
          const uint2 d = __ldg(reinterpret_cast<const uint2*>(drow) + m);
          xd[0] = bf16_lo(d.x); xd[1] = bf16_hi(d.x); xd[2] = bf16_lo(d.y); xd[3] = bf16_hi(d.y);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t v = 4 * m + e;
          xt[e] = v < e1 ? bf16_to_f32(__ldg(trow + v)) : 0.f;
          if (res) xd[e] = v < e1 ? bf16_to_f32(__ldg(drow + v)) : 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t v = 4 * m + e;
        if (v >= e1) break;
        uint32_t key;
        if (res) {
          // (p - q) / E >= 0 is finite: its bits order like the value; entries with
          // p <= q take key 0, below every candidate (if all are, the p round follows)
          const float rr = __fsub_rn(__fmul_rn(ex2(__fmaf_rn(xt[e], c, nmt)), zt),
                                     __fmul_rn(ex2(__fmaf_rn(xd[e], c, nmd)), zd));
          const float f = __uint_as_float(0x3F800000u | (ws[e] >> 9));
          const float u = __fadd_rn(__fsub_rn(f, 1.0f), 5.9604644775390625e-08f);
          key = rr > 0.f ? (__float_as_uint(__fmul_rn(rr, rcp_approx(neg_log_unit(u)))) | 0x80000000u) : 0u;
          any |= rr > 0.f ? 1 : 0;
        } else {
          key = order_key(__fadd_rn(__fmul_rn(xt[e], p.inv_t), gumbel_from_word(ws[e])));
        }
        best = umax64(best, pack_best(key, v));
      }
    }
    best = block_reduce(best, [](uint64_t a, uint64_t q) { return umax64(a, q); }, shu);
    any = block_reduce(any, [](int a, int q) { return a | q; }, shi);
    if (tid == 0) {
      part_best[round] = best;
      if (round == 0) part_any = any;
    }
    cl.sync();
  };
  sample(residual, 0);
  int any_all = 0;
  for (int q = 0; q < kEmitCtas; ++q) any_all |= *cl.map_shared_rank(&part_any, q);
  const int round = residual && !any_all ? 1 : 0;
  if (round == 1) sample(false, 1);  // uniform over the cluster
  if (r == 0 && tid == 0) {
    uint64_t best = 0ull;
    for (int q = 0; q < kEmitCtas; ++q) best = umax64(best, cl.map_shared_rank(part_best, q)[round]);
    int32_t* out = p.out_tokens + static_cast<size_t>(b) * (p.K + 1);
    for (int j = 0; j < n; ++j) out[j] = p.dtok[static_cast<size_t>(b) * p.K + j];
    out[n] = unpack_idx(best);
    for (int j = n + 1; j <= p.K; ++j) out[j] = -1;
    p.accepted[b] = n;
  }
  cl.sync();  // no CTA leaves while rank 0 reads its shared memory
}

}  // namespace

int32_t verify_launch(const uint16_t* target, const uint16_t* draft, const int32_t* dtok,
                      const uint64_t* seeds, int64_t V, int32_t bs, int32_t K, float temperature,
                      int32_t* accepted, int32_t* out_tokens, float* norms, cudaStream_t stream) {
  const float inv_t = static_cast<float>(1.0 / static_cast<double>(temperature));
  VerifyParams p{target, draft, dtok, seeds, V, bs, K, inv_t, accepted, out_tokens,
                 reinterpret_cast<float4*>(norms)};
  cudaError_t e = cudaMemsetAsync(accepted, 0, sizeof(int32_t) * static_cast<size_t>(bs), stream);
  if (e != cudaSuccess) return static_cast<int32_t>(e);
  verify_accept_kernel<<<dim3(K, bs), kVerifyThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return static_cast<int32_t>(e);
  // the sample pass as a programmatic dependent of the acceptance pass: its launch
  // overlaps the acceptance pass's end; it waits for the bits before reading them
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(kEmitCtas, bs);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int32_t>(cudaLaunchKernelEx(&cfg, verify_emit_kernel, p));
}

}  // namespace dspark
