// Per-row symmetric int8 quantization of W2 (vLLM PR #62958, "Overview": int8 W2 with
// one fp32 scale per row) and the Gumbel-noise diagnostic kernel.
//
// Quantization: one warp per row of 256 bf16 values (16 bytes per lane).
//   scale = max|w| / 127   (IEEE fp32 division)
//   q     = clamp(rint(w / scale), -127, 127)   (IEEE fp32 division, ties to even)
// An all-zero row gets scale 0 and codes 0; a non-finite entry reports
// DSPARK_ERR_NONFINITE_W2. The divisions are correctly rounded so the codes are
// reproducible bit for bit on any IEEE implementation.
#include <cstdint>

#include "common.cuh"

namespace dspark {

__global__ void __launch_bounds__(256) quantize_w2_kernel(const uint16_t* w2, int64_t V, int8_t* q,
                                                          float* scales, int32_t* status_dev) {
  const int lane = threadIdx.x & 31;
  const int64_t v = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (v >= V) return;
  const uint4 w = __ldg(reinterpret_cast<const uint4*>(w2 + v * kRank) + lane);
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  float x[8];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    x[2 * t] = bf16_lo(ww[t]);
    x[2 * t + 1] = bf16_hi(ww[t]);
  }
  float m = 0.f;
  bool finite = true;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    finite = finite && isfinite(x[t]);
    m = fmaxf(m, fabsf(x[t]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if (!__all_sync(kFull, finite) && lane == 0) report(status_dev, DSPARK_ERR_NONFINITE_W2);
  const float scale = __fdiv_rn(m, 127.f);
  uint32_t packed[2] = {0u, 0u};
  if (scale != 0.f && isfinite(scale)) {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float r = rintf(__fdiv_rn(x[t], scale));
      r = fminf(fmaxf(r, -127.f), 127.f);
      const int qi = static_cast<int>(r);
      packed[t >> 2] |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * (t & 3));
    }
  }
  reinterpret_cast<uint2*>(q + v * kRank)[lane] = make_uint2(packed[0], packed[1]);
  if (lane == 0) scales[v] = scale;
}

// Philox words and Gumbel values of every (b, i, v): one thread per 4 entries.
__global__ void gumbel_noise_kernel(const uint64_t* seeds, int bs, int K, int64_t V,
                                    uint32_t* words, float* gumbel) {
  const int64_t groups = (V + 3) / 4;
  const int64_t total = groups * bs * K;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = t % groups;
    const int64_t bi = t / groups;
    const int i = static_cast<int>(bi % K), b = static_cast<int>(bi / K);
    const uint4 w = philox_block(seeds[b], b, i, static_cast<uint32_t>(m));
    for (int j = 0; j < 4; ++j) {
      const int64_t v = 4 * m + j;
      if (v >= V) break;
      const size_t o = static_cast<size_t>(bi) * V + v;
      const uint32_t word = uint4_get(w, j);
      if (words) words[o] = word;
      if (gumbel) gumbel[o] = gumbel_from_word(word);
    }
  }
}

cudaError_t launch_quantize_w2(const uint16_t* w2, int64_t V, int8_t* q, float* scales,
                               int32_t* status_dev, cudaStream_t stream) {
  const int64_t blocks = (V + 7) / 8;
  quantize_w2_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w2, V, q, scales, status_dev);
  return cudaGetLastError();
}

cudaError_t launch_gumbel_noise(const uint64_t* seeds, int bs, int K, int64_t V, uint32_t* words,
                                float* gumbel, cudaStream_t stream) {
  const int64_t work = ((V + 3) / 4) * bs * K;
  const int64_t blocks64 = (work + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(blocks64 < 65535 * 16 ? blocks64 : 65535 * 16);
  gumbel_noise_kernel<<<blocks, 256, 0, stream>>>(seeds, bs, K, V, words, gumbel);
  return cudaGetLastError();
}

}  // namespace dspark
