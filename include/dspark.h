/*
 * dspark.h -- C ABI of the GB300 DSpark Markov draft walk (libdspark.so).
 *
 * The method (vLLM PR #62958, "Overview"; vLLM PR #49969, "Purpose"): a draft block
 * of K tokens is produced left to right. At draft position i of request row b the
 * walk forms
 *
 *     logits[b, i, :] = base_logits[b, i, :] + W2 . W1[prev_b]
 *
 * where W1 and W2 are V x rank (rank 256) and prev_b is the token chosen at the
 * previous position (at i = 0, the last accepted token), and then picks the next
 * token by argmax (greedy) or by Gumbel-max sampling at a temperature.
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; tensors are
 *     contiguous and row-major. bf16 tensors are passed as their 16-bit patterns.
 *   - Every call is asynchronous on the stream it is given and allocates nothing. A
 *     call's kernels may be launched as programmatic dependents of one another (the
 *     fused LM head's passes, the verifier's sample pass), never of the caller's
 *     kernels: work the caller enqueues after a call sees all of its results, and the
 *     calls can be captured in CUDA graphs (tested for the walk, the top-k walk, the
 *     fused LM head and the verifier).
 *   - The return value is a dspark_status code for problems found on the host
 *     (arguments, capacity, launch). Problems found on the device while the kernel
 *     runs (an out-of-range token, a wait that timed out, a non-finite W2 entry) are
 *     written to the optional device word `status_dev` (set only when non-zero;
 *     the caller zeroes it and reads it after synchronising).
 *   - Token ids are int32 (V < 2^31). Seeds are uint64, one per request row.
 *   - Ties and NaN follow torch.argmax: the first NaN wins, otherwise the first
 *     maximum (vLLM PR #64476, "New tests"); -0 and +0 are equal.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* dspark_stream_t;

typedef enum dspark_status {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,     /* null required pointer, size out of range, bad mode/T */
  DSPARK_ERR_UNSUPPORTED = 2,     /* a valid combination this library does not run */
  DSPARK_ERR_CUDA = 3,            /* a CUDA runtime call failed; see dspark_last_cuda_error */
  DSPARK_ERR_COOP_TOO_LARGE = 4,  /* the cooperative grid cannot be co-resident */
  DSPARK_ERR_TIMEOUT = 5,         /* device: a bounded wait gave up (workspace is now dirty) */
  DSPARK_ERR_BAD_TOKEN = 6,       /* device: a prev token outside [0, V); its row reads -1 */
  DSPARK_ERR_NONFINITE_W2 = 7,    /* device: quantize found a non-finite W2 entry */
  DSPARK_ERR_WORKSPACE = 8        /* workspace missing or smaller than dspark_walk_workspace_size */
} dspark_status;

typedef enum dspark_mode { DSPARK_GREEDY = 0, DSPARK_PROBABILISTIC = 1 } dspark_mode;

/* Limits of this implementation. */
#define DSPARK_RANK 256
#define DSPARK_MAX_BS 64
#define DSPARK_MAX_K 32
#define DSPARK_MAX_V 2147483647LL

/* Test and tuning knobs in dspark_walk_args.flags (0 = production behaviour). */
#define DSPARK_FLAG_SKIP_ARRIVAL_CTA0 0x1u /* CTA 0 skips its step-0 arrival: the barrier
                                              times out and the call reports TIMEOUT */
#define DSPARK_FLAG_FORCE_CUDA_CORES 0x2u  /* never use the tensor-core contraction */
#define DSPARK_FLAG_FORCE_TENSOR_CORES 0x4u /* use the tensor-core contraction for any bs */

/*
 * Arguments of one walk. Layouts:
 *   base_logits  bf16  [bs, K, V]     per-position base logits
 *   w1           bf16  [V, rank]      Markov embedding table
 *   w2           bf16  [V, rank]      Markov projection (NULL when w2q is given)
 *   w2q          int8  [V, rank]      quantized projection (from dspark_quantize_w2)
 *   w2_scales    fp32  [V]            per-row scales of w2q
 *   prev_tokens  int32 [bs]           last accepted token of each row
 *   seeds        uint64 [bs]          per-request seeds (probabilistic mode only)
 *   draft_tokens int32 [bs, K]        out: chosen tokens
 *   draft_logits bf16  [bs, K, V]     optional out: bf16(logits) that each step chose
 *                                     from (top-k: -inf off the candidates)
 *   workspace    bytes                scratch, >= dspark_walk_workspace_size(...),
 *                                     zeroed by the caller once after allocation; the
 *                                     kernels leave it zeroed again on success. After a
 *                                     TIMEOUT the caller must zero it again.
 */
typedef struct dspark_walk_args {
  const uint16_t* base_logits;
  const uint16_t* w1;
  const uint16_t* w2;
  const int8_t* w2q;
  const float* w2_scales;
  const int32_t* prev_tokens;
  const uint64_t* seeds;
  int64_t V;
  int32_t rank;        /* must be DSPARK_RANK */
  int32_t bs;          /* 1 .. DSPARK_MAX_BS */
  int32_t K;           /* 1 .. DSPARK_MAX_K */
  int32_t mode;        /* dspark_mode */
  float temperature;   /* > 0 and finite in probabilistic mode; 1.0 skips the divide */
  int32_t top_k;       /* 0: full vocabulary; 1..V: top-k walk */
  int32_t* draft_tokens;
  uint16_t* draft_logits;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status_dev; /* optional device int32 */
  uint32_t flags;      /* DSPARK_FLAG_* */
  int32_t resident_rows_cap; /* tuning: cap on smem-resident W2 rows per CTA; -1 = automatic */
  uint32_t timeout_us; /* limit of every device-side wait; 0 = 1,000,000 us */
  /* Per-request sampling settings (both optional, device memory): */
  const float* temperatures; /* fp32 [bs]: row b's temperature, overriding `temperature`;
                                a probabilistic row needs T > 0 and finite, else the walk
                                reports DSPARK_ERR_INVALID_ARG in *status_dev and writes
                                -1 for that row's tokens */
  const int32_t* row_modes;  /* int32 [bs]: row b's dspark_mode, overriding `mode` (then
                                `seeds` is required); a value other than 0 / 1 is
                                reported like an invalid temperature */
  /* Top-k walk on candidates chosen elsewhere (both optional, device memory, given
     together, top_k > 0): the candidates of every (b, i) and their base logits, e.g. from
     dspark_lmhead_topk. The walk then skips its own selection and base_logits may be
     NULL. */
  const int32_t* topk_cand;  /* int32 [bs, K, top_k] distinct vocabulary ids in [0, V), any
                                order; an id outside [0, V) is clamped into it (the walk
                                stays in bounds, its result for that (b, i) is then not a
                                walk over the given set) */
  const float* topk_base;    /* fp32 [bs, K, top_k] their base logits */
} dspark_walk_args;

/*
 * Per-row symmetric int8 quantization of W2 (vLLM PR #62958, "Overview": int8 W2 with
 * one fp32 scale per row). For each row v:
 *     scale[v] = max_k |w2[v,k]| / 127          (fp32 division)
 *     w2q[v,k] = clamp(rint(w2[v,k] / scale[v]), -127, 127)   (fp32 division, ties to even)
 * An all-zero row gets scale 0 and codes 0. A non-finite entry sets
 * DSPARK_ERR_NONFINITE_W2 in *status_dev (outputs of that row unspecified).
 *   w2         bf16 [V, rank] in;  w2q int8 [V, rank] out;  scales fp32 [V] out.
 * Returns DSPARK_ERR_INVALID_ARG for null pointers, V <= 0 or rank != DSPARK_RANK.
 */
int32_t dspark_quantize_w2(const uint16_t* w2, int64_t V, int32_t rank, int8_t* w2q,
                           float* scales, int32_t* status_dev, dspark_stream_t stream);

/*
 * The full-vocabulary walk (top_k == 0) as one persistent cooperative kernel; with
 * top_k > 0 it forwards to dspark_walk_topk. Greedy mode takes the argmax of the fp32
 * logits. Probabilistic mode takes the argmax of bf16(logit) / T + g, where
 * g = -log(-log(u)) and u comes from Philox4x32-10 with key (seed lo, seed hi) and
 * counter (v >> 2, i, b, 0), word v & 3, u = (2 * (word >> 9) + 1) * 2^-24
 * (vLLM PR #62958, "Details": Philox keyed by the request seed and draft position;
 * the sampled bf16 logits are what draft_logits holds).
 * Exactly one of w2 / (w2q, w2_scales) must be given.
 */
int32_t dspark_walk(const dspark_walk_args* args, dspark_stream_t stream);

/*
 * The top-k walk (vLLM PR #49969, "Purpose"): for every (b, i) the top_k largest base
 * logits are chosen once (NaN counts as largest; ties at the boundary go to the
 * smaller index), the bias is computed for those candidates only (bf16 W2 rows
 * gathered), and the step's argmax or sample runs over the dense row that is -inf
 * off the candidates. Gumbel noise is keyed by the vocabulary id, so top_k == V
 * reproduces dspark_walk. W2 bf16, or int8 codes with per-row scales (the gathered
 * candidate rows are then 256-byte int8 rows, the bias scale_v times their dot
 * product with the embedding).
 */
int32_t dspark_walk_topk(const dspark_walk_args* args, dspark_stream_t stream);

/*
 * The drafter's LM head fused with the top-k selection (vLLM PR #49969, "Purpose": the
 * base logits of all draft positions come from the dense LM-head output, and the top-k
 * candidates are selected from them once, before the sequential walk). For every hidden
 * row m (the (b, i) positions of a draft block, row m = b K + i) it finds the top_k
 * largest logits hidden[m] . lm_head[v] over v in [0, V) -- order: NaN largest, then
 * larger value, then smaller index -- without writing the dense [M, V] logits: a GEMM
 * over a sample of the LM-head rows sets a conservative per-row pivot, a second GEMM
 * keeps only the logits at or above it, and an exact per-row selection finishes (rows
 * the pivot did not serve take an exact path over the whole row). Logits are fp32 dot
 * products of bf16 inputs accumulated in fp32 on the tensor cores.
 *   hidden bf16 [M, d]; lm_head bf16 [V, d] (d a multiple of 64, 64..16384, both
 *   16-byte aligned); out: cand int32 [M, top_k] (any order), cand_base fp32 [M, top_k];
 *   workspace >= dspark_lmhead_workspace_size(M, V, top_k), 256-byte aligned (needs no
 *   zeroing); stats_dev optional int32 [2]: rows that took the exact path, rows whose
 *   candidate list overflowed (both counted, never reset).
 * Returns DSPARK_ERR_INVALID_ARG for null pointers, M < 1, V < 1, a bad d, top_k outside
 * 1..min(V, 8192) or misaligned tensors; DSPARK_ERR_WORKSPACE for a missing or small
 * workspace; DSPARK_ERR_CUDA if a launch fails. Device timeouts go to status_dev.
 */
typedef struct dspark_lmhead_args {
  const uint16_t* hidden;
  const uint16_t* lm_head;
  int64_t V;
  int32_t M;
  int32_t d;
  int32_t top_k;
  int32_t* cand;
  float* cand_base;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status_dev;  /* optional device int32 */
  int32_t* stats_dev;   /* optional device int32 [2] */
  uint32_t flags;       /* DSPARK_LMHEAD_FLAG_EXACT: every row takes the exact path */
  uint32_t timeout_us;  /* limit of every device-side wait; 0 = 1,000,000 us */
} dspark_lmhead_args;
#define DSPARK_LMHEAD_FLAG_EXACT 0x1u
int32_t dspark_lmhead_topk(const dspark_lmhead_args* args, dspark_stream_t stream);
/* Workspace bytes of dspark_lmhead_topk (0 for invalid sizes). */
size_t dspark_lmhead_workspace_size(int32_t M, int64_t V, int32_t top_k);

/*
 * End-to-end variant for callers whose per-call inputs live in host memory: copies
 * base_host [bs,K,V] bf16, prev_host [bs] and seeds_host [bs] (may be NULL in greedy
 * mode) into the device buffers named by `args`, runs the walk, and copies
 * draft_tokens (and draft_logits when both it and logits_host are given) back into
 * tokens_host / logits_host. All copies and the kernels are queued on `stream`; host
 * buffers should be pinned for the copies to be asynchronous. The caller synchronises.
 */
int32_t dspark_walk_from_host(const dspark_walk_args* args, const uint16_t* base_host,
                              const int32_t* prev_host, const uint64_t* seeds_host,
                              int32_t* tokens_host, uint16_t* logits_host,
                              dspark_stream_t stream);

/* Bytes of scratch workspace a walk of this shape needs (argmax slots, barrier
 * counters, status words, top-k candidate lists and their base logits). Part of the
 * walk's C interface specified with dspark_walk (caller-owned workspace, no allocation
 * in the library); the pages have no counterpart. Returns 0 for bs < 1, K < 1 or top_k < 0. */
size_t dspark_walk_workspace_size(int64_t V, int32_t bs, int32_t K, int32_t top_k);

/*
 * Part of the walk's C interface specified with dspark_walk (the shared-memory capacity
 * behind "most of W2 stays in shared memory", vLLM PR #62958, "Overview", queried at
 * run time).
 * Launch plan dspark_walk takes by default on `device` for this batch size (CUDA-core
 * contraction at bs <= 2, tensor cores from bs = 3): cooperative grid size (CTAs) and
 * the number of W2 rows kept resident in shared memory over the whole grid (greedy
 * plan; a probabilistic tensor-core walk keeps a few more). Queries
 * the device once and caches it (the only host-synchronous work of the library).
 * Returns DSPARK_ERR_INVALID_ARG for V outside 1..DSPARK_MAX_V or bs outside
 * 1..DSPARK_MAX_BS.
 */
int32_t dspark_query_capacity(int32_t device, int64_t V, int32_t w2_is_int8, int32_t bs,
                              int32_t* grid_ctas, int64_t* resident_rows);

/*
 * TEST HOOK (not needed to use the walk): the Philox words and Gumbel values the walk
 * draws, for checking them bit for bit against an independent implementation: words
 * uint32 and gumbel fp32 [bs, K, V] (either may be NULL). Same generator code as the
 * walk (vLLM PR #62958, "Details": Philox noise keyed by the request seed and the draft
 * position). Returns DSPARK_ERR_INVALID_ARG for null seeds, bs < 1, K < 1 or V <= 0.
 */
int32_t dspark_gumbel_noise(const uint64_t* seeds, int32_t bs, int32_t K, int64_t V,
                            uint32_t* words, float* gumbel, dspark_stream_t stream);

/*
 * dspark_walk without a caller-provided workspace, for callers that cannot allocate
 * device memory (e.g. a plugin whose enqueue hook may not call cudaMalloc, or a server
 * whose device memory is all pre-reserved by a caching allocator; cudaMalloc on the
 * decode path would fail or synchronise). The pages have no counterpart of this call.
 *   - Takes the same arguments as dspark_walk; `workspace` and `workspace_bytes` are
 *     ignored. Invalid arguments return DSPARK_ERR_INVALID_ARG before any CUDA call
 *     (the same checks as dspark_walk); then, full-vocabulary walk only: a valid
 *     top_k > 0 returns DSPARK_ERR_UNSUPPORTED.
 *   - Scratch comes from one static device array of 24,576 bytes inside the library,
 *     held by every GPU that loads the library until the process exits. A shape whose
 *     scratch would not fit returns DSPARK_ERR_WORKSPACE (every shape dspark_walk
 *     accepts fits).
 *   - The first call on a device looks up the array's device address with that device
 *     current. With CUDA's lazy module loading (the default) that lookup also loads
 *     this part of the library onto the device, which creates the array's storage
 *     then: make the first call on each device at start-up, before the caller hands
 *     its device memory to a caching allocator and before any stream capture.
 *   - Each call clears the part of the array it uses with cudaMemsetAsync on `stream`,
 *     then launches the walk; it calls no allocating routine. All calls share the
 *     array, so calls whose kernels overlap on the GPU (different streams, no ordering)
 *     race and give wrong results: serialise them.
 */
int32_t dspark_walk_noalloc(const dspark_walk_args* args, dspark_stream_t stream);

/*
 * Speculative-sampling verification of drafted tokens (Leviathan, Kalman, Matias, ICML
 * 2023, Algorithm 1), consuming the walk's draft_logits, which are the distribution the
 * draft tokens were sampled from (vLLM PR #62958, "Details"). With
 * q_i = softmax(draft_logits[b, i, :] / T) and p_i = softmax(target_logits[b, i, :] / T):
 * draft i is accepted iff u_i q_i(d_i) < p_i(d_i); at the first rejection a sample of
 * norm(max(0, p_i - q_i)) is emitted and the row stops; if all K are accepted a sample
 * of p_K is emitted. Samples are Gumbel-max draws: the argmax over v of
 * log(p(v) - q(v)) + g_v where p > q (if p > q nowhere after rounding, the scores of
 * p), and of target[b, K, v] / T + g_v for the bonus token. u_i = (2 (w >> 9) + 1) 2^-24
 * and g_v = -log(-log u_v) come from the walk's Philox4x32-10 keyed by the row's seed,
 * counter (0, i, b, 1), word 0, for u_i, and (v >> 2, n, b, 2), word v & 3, for the
 * noise at the emitting position n (the walk uses counter word 3 = 0), so the
 * verification is reproducible and never reuses the drafter's noise.
 *   target_logits bf16 [bs, K+1, V]; draft_logits bf16 [bs, K, V]; draft_tokens int32
 *   [bs, K]; seeds uint64 [bs]; out: accepted int32 [bs] (0..K), out_tokens int32
 *   [bs, K+1] (the accepted drafts, the emitted sample, then -1). All device memory
 *   owned by the caller; asynchronous on `stream`. A draft token outside [0, V) is
 *   rejected. No alignment is required (16- and 8-byte loads are used where the rows
 *   allow them). norms (optional, caller-owned scratch, fp32 [bs, K, 4], 16-byte
 *   aligned): the acceptance pass leaves there the softmax normalisers (running
 *   maximum, sum) of the target and draft rows of every (row, position), and the
 *   sample pass reads those of the emitting position instead of recomputing them over
 *   the two rows; with NULL they are recomputed (the same values up to the summation
 *   order). Returns DSPARK_ERR_INVALID_ARG for null pointers, V outside
 *   1..DSPARK_MAX_V, bs outside 1..DSPARK_MAX_BS, K outside 1..DSPARK_MAX_K, T not
 *   > 0 and finite, or norms not 16-byte aligned; DSPARK_ERR_CUDA if a launch fails.
 */
typedef struct dspark_verify_args {
  const uint16_t* target_logits;
  const uint16_t* draft_logits;
  const int32_t* draft_tokens;
  const uint64_t* seeds;
  int64_t V;
  int32_t bs;
  int32_t K;
  float temperature;
  int32_t* accepted;
  int32_t* out_tokens;
  float* norms;        /* optional scratch fp32 [bs, K, 4], 16-byte aligned, or NULL */
} dspark_verify_args;
int32_t dspark_verify(const dspark_verify_args* args, dspark_stream_t stream);

/* Human-readable name of a status code (static storage). Part of the C interface's
 * error reporting; the pages have no counterpart. */
const char* dspark_status_string(int32_t status);

/* The last CUDA error string seen by this thread's calls into the library (for
 * DSPARK_ERR_CUDA, and the reason of a DSPARK_ERR_UNSUPPORTED launch refusal). Part of
 * the C interface's error reporting; the pages have no counterpart. */
const char* dspark_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H_ */
