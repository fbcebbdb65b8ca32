// CPU oracle for the DSpark Markov draft walk.
//
// TEST INFRASTRUCTURE ONLY. Plain, slow and meant to be checked by eye against the
// method's definition. Only the test suite, the package's smoke check and the
// benchmark's CPU-baseline leg may load this library; the product path never does.
// It shares no code, header, table or helper with the CUDA path.
//
// Sources (vLLM pull-request pages describing the method):
//   * vLLM PR #62958 (int8 cooperative Markov walk), "Overview": each draft position
//     adds the Markov bias W2 . W1[prev] (W2 is V x 256) to that position's base
//     logits and then takes an argmax or a sample; the chosen token becomes `prev`
//     of the next position. Same page: W2 may be int8 with one fp32 scale per row.
//   * vLLM PR #62958, "Details": probabilistic drafting samples from bf16 logits
//     that are cached as draft_logits; Philox noise is keyed by the request seed and
//     the draft position.
//   * vLLM PR #64476 (Markov sampling in the Gumbel kernel), "Claims" and "New tests":
//     the temperature divide is skipped at 1.0; ties and NaN follow torch.argmax
//     (the first NaN wins, otherwise the first maximum).
//   * vLLM PR #49969 ([Spec Decode] Add top-k DSpark Markov projection), "Purpose":
//     top-k candidates are chosen once from the base logits of each position; the
//     bias is applied to those candidates only and scattered into a row that is
//     -inf everywhere else; the unchanged sampler then runs on that dense row.
//   * Philox4x32-10: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
//     Random Numbers: As Easy as 1, 2, 3", SC'11.
//
// Readings where the pages are silent:
//   * quantizer: scale = max|w| / 127 in fp32; q = round-half-even(w / scale) in fp32,
//     clamped to [-127, 127]; an all-zero row has scale 0 and q = 0.
//   * the probabilistic score is bf16(l) / T + g with g = -log(-log(u)); greedy uses l.
//   * Philox counter = (v >> 2, i, b, 0), key = (seed low 32 bits, seed high 32 bits),
//     word = output[v & 3], u = (2 * (word >> 9) + 1) * 2^-24.
//   * top-k order: NaN largest, then larger value, then smaller index; -0 == +0.
//
// Arithmetic: fp64 accumulation in sequential k order; compiled with
// -O2 -ffp-contract=off and without fast-math. An optional OpenMP loop over the
// vocabulary leaves the arithmetic of every element unchanged.

#include <algorithm>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum {
  ORACLE_OK = 0,
  ORACLE_INVALID_ARG = 1,
  ORACLE_UNSUPPORTED = 2,
  ORACLE_BAD_TOKEN = 6,
  ORACLE_NONFINITE_W2 = 7,
};

float bf16_bits_to_float(uint16_t h) {
  uint32_t bits = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

double bf16_bits_to_double(uint16_t h) { return static_cast<double>(bf16_bits_to_float(h)); }

// Round a binary64 value to the nearest bfloat16 (8 exponent bits, 7 stored fraction
// bits), ties to even, in one rounding step.
uint16_t round_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  if (std::isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  int e = 0;
  std::frexp(std::fabs(x), &e);  // |x| = f * 2^e with f in [0.5, 1)
  int binade = e - 1;            // floor(log2 |x|)
  if (binade < -126) binade = -126;  // subnormals keep the spacing of the lowest normal binade
  const double quantum = std::ldexp(1.0, binade - 7);
  const double r = std::nearbyint(x / quantum) * quantum;  // FE_TONEAREST: ties to even
  if (std::fabs(r) >= std::ldexp(1.0, 128)) return x > 0 ? 0x7F80 : 0xFF80;
  const float f = static_cast<float>(r);  // exact: r has <= 8 significant bits
  uint32_t bits;
  std::memcpy(&bits, &f, sizeof bits);
  return static_cast<uint16_t>(bits >> 16);
}

// Philox4x32-10 (SC'11): ten rounds of the 4x32 bijection; round r uses the key
// bumped r times by the Weyl constants.
void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    const uint64_t p0 = static_cast<uint64_t>(M0) * x0;
    const uint64_t p1 = static_cast<uint64_t>(M1) * x2;
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    const uint32_t y0 = hi1 ^ x1 ^ k0;
    const uint32_t y1 = lo1;
    const uint32_t y2 = hi0 ^ x3 ^ k1;
    const uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// Counter (v >> 2, i, b, domain), word v & 3. Domain 0: the drafter's Gumbel noise;
// 1: the verifier's acceptance uniforms (v = 0); 2: the verifier's resampling noise.
uint32_t philox_word(uint64_t seed, int32_t b, int32_t i, int64_t v, uint32_t domain = 0u) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(i),
                           static_cast<uint32_t>(b), domain};
  const uint32_t key[2] = {static_cast<uint32_t>(seed & 0xFFFFFFFFull),
                           static_cast<uint32_t>(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return out[v & 3];
}

// u = (2 * (word >> 9) + 1) * 2^-24: the odd multiples of 2^-24 in (0, 1), exact in fp32.
float uniform_from_word(uint32_t w) {
  const float odd = static_cast<float>(2u * (w >> 9) + 1u);
  return odd * 0x1p-24f;
}

double gumbel(uint64_t seed, int32_t b, int32_t i, int64_t v) {
  const double u = static_cast<double>(uniform_from_word(philox_word(seed, b, i, v)));
  return -std::log(-std::log(u));
}

// The verifier's resampling noise (counter domain 2).
double gumbel_d(uint64_t seed, int32_t b, int32_t i, int64_t v) {
  const double u = static_cast<double>(uniform_from_word(philox_word(seed, b, i, v, 2u)));
  return -std::log(-std::log(u));
}

// torch.argmax order on a row of scores: the first NaN if any, else the first maximum.
int64_t argmax_first(const std::vector<double>& s) {
  int64_t best = 0;
  if (std::isnan(s[0])) return 0;
  for (int64_t v = 1; v < static_cast<int64_t>(s.size()); ++v) {
    if (std::isnan(s[v])) return v;
    if (s[v] > s[best]) best = v;
  }
  return best;
}

// Score gap between the winner and the best other entry; +inf when the winner is NaN
// or strictly beats an infinite runner-up; 0 for an exact tie.
double top2_gap(const std::vector<double>& s, int64_t best) {
  if (std::isnan(s[best])) return std::numeric_limits<double>::infinity();
  double second = -std::numeric_limits<double>::infinity();
  bool have_second = false;
  for (int64_t v = 0; v < static_cast<int64_t>(s.size()); ++v) {
    if (v == best || std::isnan(s[v])) continue;
    if (!have_second || s[v] > second) { second = s[v]; have_second = true; }
  }
  if (!have_second) return std::numeric_limits<double>::infinity();
  if (s[best] == second) return 0.0;
  const double g = s[best] - second;
  return std::isnan(g) ? 0.0 : g;
}

// Top-k order for the candidate selection: NaN first (NaNs by index), then larger
// value, then smaller index. -0 and +0 compare equal.
bool topk_before(double a, int64_t ia, double b, int64_t ib) {
  const bool na = std::isnan(a), nb = std::isnan(b);
  if (na != nb) return na;
  if (na && nb) return ia < ib;
  if (a != b) return a > b;
  return ia < ib;
}

}  // namespace

extern "C" {

struct oracle_walk_args {
  const uint16_t* base;      // [bs, K, V] bf16 bit patterns
  const uint16_t* w1;        // [V, R] bf16
  const uint16_t* w2;        // [V, R] bf16, or null when w2q is given
  const int8_t* w2q;         // [V, R] int8, or null
  const float* w2_scales;    // [V] fp32 (with w2q)
  const int32_t* prev;       // [bs] last accepted token of each row
  const uint64_t* seeds;     // [bs] per-request seeds (probabilistic mode)
  const int32_t* slot;       // [bs] batch slot b used in the Philox counter, or null (= row)
  int64_t V;
  int32_t R, bs, K, mode;    // mode: 0 greedy, 1 probabilistic
  float temperature;
  int32_t top_k;             // 0 = full vocabulary
  const int32_t* follow;     // [bs, K] tokens to continue with when acceptable, or null
  double tie_tol;            // acceptance window for `follow` tokens (score units)
  double bf16_eps;           // |l - bf16 midpoint| window for the bf16-boundary class
  int32_t nthreads;          // OpenMP threads for the vocabulary loop (<= 0: 1)
  // outputs (all optional except tokens)
  int32_t* tokens;           // [bs, K] the oracle's own argmax at each step
  double* gap;               // [bs, K] top-2 score gap at each step
  double* best_score;        // [bs, K]
  uint8_t* follow_class;     // [bs, K] 0 same, 1 near-tie, 2 bf16-boundary, 255 rejected
  double* logits;            // [bs, K, V] fp64 logits (-inf off the top-k candidates)
  uint16_t* logits_bf16;     // [bs, K, V] bf16(l)
  double* scores;            // [bs, K, V] scores the argmax ran over
  int32_t* cand;             // [bs, K, top_k] candidates in ascending vocabulary order
  const double* base_f64;    // optional [bs, K, V] base logits in fp64 (unrounded), used
                             // instead of `base` when given (the drafter's LM-head output)
};

double oracle_bf16_to_double(uint16_t h) { return bf16_bits_to_double(h); }

uint16_t oracle_round_bf16(double x) {
  std::fesetround(FE_TONEAREST);
  return round_to_bf16(x);
}

void oracle_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}

// Philox word, uniform and Gumbel value for each (b, i, v) of a [bs, K, V] block.
void oracle_gumbel_block(const uint64_t* seeds, int32_t bs, int32_t K, int64_t V,
                         uint32_t* words, float* uniforms, double* g) {
  for (int32_t b = 0; b < bs; ++b)
    for (int32_t i = 0; i < K; ++i)
      for (int64_t v = 0; v < V; ++v) {
        const int64_t o = (static_cast<int64_t>(b) * K + i) * V + v;
        const uint32_t w = philox_word(seeds[b], b, i, v);
        const float u = uniform_from_word(w);
        if (words) words[o] = w;
        if (uniforms) uniforms[o] = u;
        if (g) g[o] = -std::log(-std::log(static_cast<double>(u)));
      }
}

// Per-row symmetric int8 quantization of a bf16 [V, R] matrix.
int32_t oracle_quantize_w2(const uint16_t* w2, int64_t V, int32_t R, int8_t* q, float* scales) {
  if (!w2 || !q || !scales || V <= 0 || R <= 0) return ORACLE_INVALID_ARG;
  std::fesetround(FE_TONEAREST);
  int32_t status = ORACLE_OK;
  for (int64_t v = 0; v < V; ++v) {
    const uint16_t* row = w2 + v * R;
    float m = 0.0f;
    for (int32_t k = 0; k < R; ++k) {
      const float x = bf16_bits_to_float(row[k]);
      if (!std::isfinite(x)) status = ORACLE_NONFINITE_W2;
      const float a = std::fabs(x);
      if (a > m) m = a;
    }
    const float scale = m / 127.0f;
    scales[v] = scale;
    for (int32_t k = 0; k < R; ++k) {
      int8_t out = 0;
      if (scale != 0.0f && std::isfinite(scale)) {
        const float x = bf16_bits_to_float(row[k]);
        float r = std::nearbyint(x / scale);
        if (!(r >= -127.0f)) r = -127.0f;  // also catches NaN
        if (r > 127.0f) r = 127.0f;
        out = static_cast<int8_t>(r);
      }
      q[v * R + k] = out;
    }
  }
  return status;
}

// Top-k candidate set of one fp64 row (the same order: NaN first, then larger value,
// then smaller index), ascending vocabulary order.
void topk_select_f64(const double* row, int64_t V, int32_t k, int32_t* cand) {
  std::vector<int64_t> order(V);
  for (int64_t v = 0; v < V; ++v) order[v] = v;
  std::partial_sort(order.begin(), order.begin() + k, order.end(),
                    [&](int64_t a, int64_t b) { return topk_before(row[a], a, row[b], b); });
  std::vector<int64_t> chosen(order.begin(), order.begin() + k);
  std::sort(chosen.begin(), chosen.end());
  for (int32_t j = 0; j < k; ++j) cand[j] = static_cast<int32_t>(chosen[j]);
}

// The drafter's LM head (vLLM PR #49969, "Purpose": the base logits of every draft
// position come from the dense LM-head output): logits[m, v] = sum_k hidden[m, k] *
// lm_head[v, k] in fp64, sequential k order, unrounded.
int32_t oracle_lmhead_logits(const uint16_t* hidden, const uint16_t* lm_head, int32_t M, int32_t d,
                             int64_t V, double* out, int32_t nthreads) {
  if (!hidden || !lm_head || !out || M <= 0 || d <= 0 || V <= 0) return ORACLE_INVALID_ARG;
#ifdef _OPENMP
  const int nt = nthreads > 0 ? nthreads : 1;
#else
  (void)nthreads;
#endif
  for (int32_t m = 0; m < M; ++m) {
    std::vector<double> h(d);
    for (int32_t k = 0; k < d; ++k) h[k] = bf16_bits_to_double(hidden[static_cast<int64_t>(m) * d + k]);
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(static)
#endif
    for (int64_t v = 0; v < V; ++v) {
      const uint16_t* w = lm_head + v * d;
      double acc = 0.0;
      for (int32_t k = 0; k < d; ++k) acc += h[k] * bf16_bits_to_double(w[k]);
      out[static_cast<int64_t>(m) * V + v] = acc;
    }
  }
  return ORACLE_OK;
}

// Top-k candidate set of every (b, i) row of the base logits, ascending vocab order.
int32_t oracle_topk_select(const uint16_t* base, int32_t rows, int64_t V, int32_t k,
                           int32_t* cand) {
  if (!base || !cand || rows <= 0 || V <= 0 || k <= 0 || k > V) return ORACLE_INVALID_ARG;
  std::vector<int64_t> order(V);
  for (int32_t r = 0; r < rows; ++r) {
    const uint16_t* row = base + static_cast<int64_t>(r) * V;
    for (int64_t v = 0; v < V; ++v) order[v] = v;
    std::partial_sort(order.begin(), order.begin() + k, order.end(),
                      [&](int64_t a, int64_t b) {
                        return topk_before(bf16_bits_to_double(row[a]), a,
                                           bf16_bits_to_double(row[b]), b);
                      });
    std::vector<int64_t> chosen(order.begin(), order.begin() + k);
    std::sort(chosen.begin(), chosen.end());
    for (int32_t j = 0; j < k; ++j) cand[static_cast<int64_t>(r) * k + j] = static_cast<int32_t>(chosen[j]);
  }
  return ORACLE_OK;
}

// The K-step walk of every row, in the order the method defines it.
int32_t oracle_walk(const oracle_walk_args* a) {
  if (!a || (!a->base && !a->base_f64) || !a->w1 || !a->prev || !a->tokens) return ORACLE_INVALID_ARG;
  if (a->V <= 0 || a->R <= 0 || a->bs <= 0 || a->K <= 0) return ORACLE_INVALID_ARG;
  if (a->mode != 0 && a->mode != 1) return ORACLE_INVALID_ARG;
  const bool int8_w2 = a->w2 == nullptr;
  if (int8_w2 && (!a->w2q || !a->w2_scales)) return ORACLE_INVALID_ARG;
  if (a->mode == 1 && (!a->seeds || !(a->temperature > 0.0f) || !std::isfinite(a->temperature)))
    return ORACLE_INVALID_ARG;
  if (a->top_k < 0 || a->top_k > a->V) return ORACLE_INVALID_ARG;
  std::fesetround(FE_TONEAREST);
#ifdef _OPENMP
  const int nthreads = a->nthreads > 0 ? a->nthreads : 1;
#endif

  const int64_t V = a->V;
  const int32_t R = a->R, K = a->K;
  const double T = static_cast<double>(a->temperature);
  const double ninf = -std::numeric_limits<double>::infinity();
  int32_t status = ORACLE_OK;

  std::vector<double> e(R), l(V), s(V);
  std::vector<uint8_t> is_cand;
  std::vector<int32_t> cand_row(a->top_k > 0 ? a->top_k : 0);

  for (int32_t row = 0; row < a->bs; ++row) {
    const int32_t b = a->slot ? a->slot[row] : row;
    int64_t prev = a->prev[row];
    bool diverged = false;
    if (prev < 0 || prev >= V) {
      status = ORACLE_BAD_TOKEN;
      for (int32_t i = 0; i < K; ++i) {
        a->tokens[static_cast<int64_t>(row) * K + i] = -1;
        if (a->follow_class) a->follow_class[static_cast<int64_t>(row) * K + i] = 255;
      }
      continue;
    }
    for (int32_t i = 0; i < K; ++i) {
      const int64_t ri = static_cast<int64_t>(row) * K + i;
      const uint16_t* base_row = a->base ? a->base + ri * V : nullptr;
      const double* base_row64 = a->base_f64 ? a->base_f64 + ri * V : nullptr;
      auto base_at = [&](int64_t v) { return base_row64 ? base_row64[v] : bf16_bits_to_double(base_row[v]); };

      // The Markov embedding of the previous token.
      for (int32_t k = 0; k < R; ++k) e[k] = bf16_bits_to_double(a->w1[prev * R + k]);

      // Top-k: candidates chosen once per position from the unbiased base logits.
      if (a->top_k > 0) {
        if (base_row64) topk_select_f64(base_row64, V, a->top_k, cand_row.data());
        else oracle_topk_select(base_row, 1, V, a->top_k, cand_row.data());
        is_cand.assign(V, 0);
        for (int32_t j = 0; j < a->top_k; ++j) is_cand[cand_row[j]] = 1;
        if (a->cand)
          for (int32_t j = 0; j < a->top_k; ++j) a->cand[ri * a->top_k + j] = cand_row[j];
      }

      // Bias, logit and score of every vocabulary entry.
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(static)
#endif
      for (int64_t v = 0; v < V; ++v) {
        double lv;
        if (a->top_k > 0 && !is_cand[v]) {
          lv = ninf;
        } else {
          double bias = 0.0;
          if (int8_w2) {
            const int8_t* qrow = a->w2q + v * R;
            double acc = 0.0;
            for (int32_t k = 0; k < R; ++k) acc += static_cast<double>(qrow[k]) * e[k];
            bias = static_cast<double>(a->w2_scales[v]) * acc;
          } else {
            const uint16_t* wrow = a->w2 + v * R;
            for (int32_t k = 0; k < R; ++k) bias += bf16_bits_to_double(wrow[k]) * e[k];
          }
          lv = base_at(v) + bias;
        }
        l[v] = lv;
        if (a->mode == 0) {
          s[v] = lv;
        } else {
          const double lb = bf16_bits_to_double(round_to_bf16(lv));
          s[v] = lb / T + gumbel(a->seeds[row], b, i, v);
        }
      }

      const int64_t tok = argmax_first(s);
      a->tokens[ri] = static_cast<int32_t>(tok);
      if (a->gap) a->gap[ri] = top2_gap(s, tok);
      if (a->best_score) a->best_score[ri] = s[tok];
      if (a->logits) std::memcpy(a->logits + ri * V, l.data(), sizeof(double) * V);
      if (a->logits_bf16)
        for (int64_t v = 0; v < V; ++v) a->logits_bf16[ri * V + v] = round_to_bf16(l[v]);
      if (a->scores) std::memcpy(a->scores + ri * V, s.data(), sizeof(double) * V);

      // Next step's previous token: the oracle's own pick, or an acceptable `follow` token.
      int64_t next = tok;
      if (a->follow) {
        const int64_t f = a->follow[ri];
        uint8_t cls = 255;
        if (!diverged && f >= 0 && f < V) {
          if (f == tok) {
            cls = 0;
          } else if (!std::isnan(s[tok]) && !std::isnan(s[f]) && s[f] >= s[tok] - a->tie_tol) {
            cls = 1;
          } else if (a->mode == 1 && !std::isnan(s[tok]) && !std::isnan(s[f]) &&
                     std::isfinite(l[f]) && std::isfinite(l[tok])) {
            // The sampled logit is rounded to bf16. A logit within bf16_eps of a rounding
            // midpoint may round the other way in fp32; score both candidates with the
            // rounding that favours `f` and accept if `f` then comes within tie_tol.
            auto alt_score = [&](int64_t v, bool up) {
              const double lb = bf16_bits_to_double(round_to_bf16(l[v]));
              const double lo = bf16_bits_to_double(round_to_bf16(l[v] - a->bf16_eps));
              const double hi = bf16_bits_to_double(round_to_bf16(l[v] + a->bf16_eps));
              const double pick = up ? std::max(lb, hi) : std::min(lb, lo);
              return pick / T + gumbel(a->seeds[row], b, i, v);
            };
            if (alt_score(f, true) >= alt_score(tok, false) - a->tie_tol) cls = 2;
          }
        }
        if (a->follow_class) a->follow_class[ri] = cls;
        if (cls != 255) next = f; else diverged = true;
      }
      prev = next;
    }
  }
  return status;
}

// ---------------------------------------------------------------- verification
//
// Speculative sampling verification of K drafted tokens (Leviathan, Kalman, Matias,
// "Fast Inference from Transformers via Speculative Decoding", ICML 2023, Algorithm 1;
// Chen et al., "Accelerating Large Language Model Decoding with Speculative Sampling",
// 2023), consuming the draft_logits the walk kept (vLLM PR #62958, "Details": the bf16
// draft logits are the distribution the draft tokens were sampled from).
//   q_i = softmax(draft[b, i, :] / T), p_i = softmax(target[b, i, :] / T);
//   for i = 0 .. K-1: u_i uniform (domain 1); accept d_i iff u_i q_i(d_i) < p_i(d_i);
//     at the first rejection emit a sample of norm(max(0, p_i - q_i)) and stop;
//   all accepted: emit a sample of p_K.
// Samples by Gumbel-max with domain-2 noise: residual scores log(p - q) + g where
// p > q (if p > q nowhere, the scores of p: target / T + g), bonus target / T + g.
struct oracle_verify_args {
  const uint16_t* target;    // [bs, K+1, V] bf16 target logits
  const uint16_t* draft;     // [bs, K, V] bf16 draft logits
  const int32_t* dtok;       // [bs, K] draft tokens
  const uint64_t* seeds;     // [bs]
  const int32_t* slot;       // [bs] batch slot b in the Philox counter, or null (= row)
  int64_t V;
  int32_t bs, K;
  float temperature;
  int32_t* accepted;         // [bs] accepted draft tokens
  int32_t* out_tokens;       // [bs, K+1] accepted drafts, the emitted sample, then -1
  double* p_out;             // optional [bs, K+1, V] target probabilities
  double* q_out;             // optional [bs, K, V] draft probabilities
  double* u_out;             // optional [bs, K] acceptance uniforms
  double* ratio_out;         // optional [bs, K] p_i(d_i) and q_i(d_i): ratio_out = p, qd_out = q
  double* qd_out;            // optional [bs, K]
  int32_t* y_out;            // optional [bs, K+1] the sample of every position (residual / bonus)
  double* gap_out;           // optional [bs, K+1] its top-2 score gap
  double* score_out;         // optional [bs, K+1, V] the sampling scores
};

int32_t oracle_verify(const oracle_verify_args* a) {
  if (!a || !a->target || !a->draft || !a->dtok || !a->seeds || !a->accepted || !a->out_tokens)
    return ORACLE_INVALID_ARG;
  if (a->V <= 0 || a->bs <= 0 || a->K <= 0 || !(a->temperature > 0.0f) || !std::isfinite(a->temperature))
    return ORACLE_INVALID_ARG;
  const int64_t V = a->V;
  const int32_t K = a->K;
  const double T = static_cast<double>(a->temperature);
  const double ninf = -std::numeric_limits<double>::infinity();
  std::vector<double> p(V), q(V), s(V);
  // softmax of a bf16 row divided by T (all zero when the row is -inf everywhere)
  auto softmax = [&](const uint16_t* row, std::vector<double>& out) {
    double m = ninf;
    for (int64_t v = 0; v < V; ++v) m = std::max(m, bf16_bits_to_double(row[v]) / T);
    double z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      out[v] = m == ninf ? 0.0 : std::exp(bf16_bits_to_double(row[v]) / T - m);
      z += out[v];
    }
    for (int64_t v = 0; v < V; ++v) out[v] = z > 0.0 ? out[v] / z : 0.0;
  };
  for (int32_t r = 0; r < a->bs; ++r) {
    const int32_t b = a->slot ? a->slot[r] : r;
    const uint64_t seed = a->seeds[r];
    int32_t n_acc = -1;  // first rejected position, -1 while all accepted
    for (int32_t i = 0; i <= K; ++i) {
      const uint16_t* trow = a->target + (static_cast<size_t>(r) * (K + 1) + i) * V;
      softmax(trow, p);
      if (a->p_out) std::copy(p.begin(), p.end(), a->p_out + (static_cast<size_t>(r) * (K + 1) + i) * V);
      bool residual = false;
      if (i < K) {
        softmax(a->draft + (static_cast<size_t>(r) * K + i) * V, q);
        if (a->q_out) std::copy(q.begin(), q.end(), a->q_out + (static_cast<size_t>(r) * K + i) * V);
        const int32_t d = a->dtok[static_cast<size_t>(r) * K + i];
        const double u = static_cast<double>(uniform_from_word(philox_word(seed, b, i, 0, 1u)));
        const double pd = (d >= 0 && d < V) ? p[d] : 0.0, qd = (d >= 0 && d < V) ? q[d] : 0.0;
        if (a->u_out) a->u_out[static_cast<size_t>(r) * K + i] = u;
        if (a->ratio_out) a->ratio_out[static_cast<size_t>(r) * K + i] = pd;
        if (a->qd_out) a->qd_out[static_cast<size_t>(r) * K + i] = qd;
        if (n_acc < 0 && !(u * qd < pd)) n_acc = i;
        for (int64_t v = 0; v < V; ++v) {
          const double rv = p[v] - q[v];
          s[v] = rv > 0.0 ? std::log(rv) + gumbel_d(seed, b, i, v) : ninf;
          residual = residual || rv > 0.0;
        }
      }
      if (!residual)  // bonus position, or p > q nowhere: a sample of p
        for (int64_t v = 0; v < V; ++v) s[v] = bf16_bits_to_double(trow[v]) / T + gumbel_d(seed, b, i, v);
      const int64_t y = argmax_first(s);
      if (a->y_out) a->y_out[static_cast<size_t>(r) * (K + 1) + i] = static_cast<int32_t>(y);
      if (a->gap_out) a->gap_out[static_cast<size_t>(r) * (K + 1) + i] = top2_gap(s, y);
      if (a->score_out) std::copy(s.begin(), s.end(), a->score_out + (static_cast<size_t>(r) * (K + 1) + i) * V);
      const int32_t n = n_acc < 0 ? K : n_acc;
      if (i == n) {  // the emitted sample (first rejection, or the bonus)
        int32_t* out = a->out_tokens + static_cast<size_t>(r) * (K + 1);
        for (int32_t j = 0; j < n; ++j) out[j] = a->dtok[static_cast<size_t>(r) * K + j];
        out[n] = static_cast<int32_t>(y);
        for (int32_t j = n + 1; j <= K; ++j) out[j] = -1;
        a->accepted[r] = n;
      }
    }
  }
  return ORACLE_OK;
}

}  // extern "C"
