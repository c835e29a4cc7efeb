/*
 * dsample.h -- C ABI of libdsample, the GB300 (sm_103a) vocab-wide sampling pass.
 *
 * The two hot-path calls:
 *
 *   ds_sample      classifier-free-guidance combine, full-vocab max / logsumexp,
 *                  exact top-ratio filter and Gumbel-max sampling at per-request
 *                  temperature; one (token, logprob) per (row, position) cell.
 *   ds_greedy_lse  per-row max, logsumexp and argmax over a large vocabulary.
 *
 * and the calls around them: ds_sample_ex (per-request ratios and iterations,
 * keep-ties mode), ds_reveal (confidence ranking and reveal), ds_merge_triples
 * (vocabulary-shard merge) and ds_log_softmax (dense log-probabilities). All are
 * asynchronous on the caller's CUDA stream, allocate nothing and keep no state
 * between calls beyond a process-wide count of kernel launches
 * (ds_launch_count).
 *
 * All pointers named "device" must be CUDA device (or managed) memory of the
 * current device; the library never frees or retains them. Inputs are never
 * written. The stream argument is a cudaStream_t (NULL = legacy default
 * stream). A host-side error is returned synchronously and nothing is
 * launched; errors that only the GPU can see are reported through the
 * optional device status word (see ds_sample).
 */
#ifndef DSAMPLE_H
#define DSAMPLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad scalar */
  DS_ERR_UNSUPPORTED = 2, /* valid but outside what this build supports (see limits) */
  DS_ERR_CUDA = 3         /* a CUDA runtime call or the kernel launch failed */
} ds_status;

/* Bits OR-ed into *d_status by the kernels (device-detected input errors). */
#define DS_DEV_ERR_LAYOUT 1u   /* sum(seq_lens) != P, or a negative seq_len */
#define DS_DEV_ERR_NO_UNCOND 2u /* guidance != 0 for a request but u_logits == NULL */
#define DS_DEV_ERR_PARAM 4u    /* temperature < 0 or NaN, or guidance NaN */

/* Limits of this build. */
#define DS_MAX_ROWS 256          /* C: rows (codebooks) per call; the row index keys the noise */
#define DS_MAX_ITERATION 16777215u /* iteration < 2^24; it keys the noise next to the row */
#define DS_MAX_VOCAB 524281      /* largest V of ds_sample (16-CTA cluster, 32K elements per CTA) */

/*
 * ds_sample -- sample every cell of a packed batch of guided logits.
 *
 * Defined by: "Sampler support for discrete diffusion" (mstar issue #267),
 * Hert4's first comment (log-softmax, argmax and confidence per cell; logits
 * [C, T, V] with T ragged across requests; CFG combine of two logit tensors;
 * top-ratio filter keeping ceil(0.1 * V); Gumbel sampling; the sampler returns
 * a (token, logprob) for every position it is given and leaves ranking to the
 * caller), and "Add a sampler resource
 * for discrete diffusion" (mstar PR #290), Contract (sample(request_ids,
 * c_logits, u_logits, seq_lens, iterations) over [rows, positions, vocab]
 * packed across requests; per-request guidance and temperature; no
 * unconditional document at guidance 0).
 *
 * Arguments (B requests, C rows, P = sum of seq_lens positions, V vocabulary):
 *   request_ids  device int32 [B]; any values; they key the noise of a request.
 *   c_logits     device bf16 [C][P][V], V contiguous; request r owns positions
 *                [off_r, off_r + seq_lens[r]) with off_r = sum_{j<r} seq_lens[j].
 *                Needs 2-byte alignment only; rows may start anywhere.
 *   u_logits     device bf16 [C][P_u][V], the unconditional logits of the
 *                requests with guidance != 0 only, packed in request order
 *                (P_u = sum of their seq_lens). NULL when no request is guided.
 *   seq_lens     device int32 [B], each >= 0, summing to P.
 *   B, C, P, V   B >= 0, 0 <= C <= DS_MAX_ROWS, P >= 0, 1 <= V <= DS_MAX_VOCAB.
 *                C == 0 or P == 0 is a valid empty call (nothing launched).
 *   guidance     device float [B]; per-request guidance g; z = c + g (c - u) in
 *                fp32 (difference rounded, then one fma); g == 0 reads no u.
 *   temperature  device float [B]; tau >= 0; tau == 0 returns the argmax.
 *   top_ratio    (0, 1]; the kept set is the k = ceilf(top_ratio * V) largest z
 *                (product in fp32, k clamped to [1, V]), ties at the cut kept
 *                by smallest id.
 *   seed         Philox4x32-10 key (low word, high word).
 *   iteration    < 2^24; the denoising step; it keys the noise.
 *   out_tokens   device int32 [C][P]: sampled token, argmax when tau == 0;
 *                ties between equal perturbed scores go to the smallest id.
 *   out_logprobs device float [C][P]: z[token] - logsumexp(z) over the full,
 *                unfiltered, untempered vocabulary.
 *   d_status     device uint32 word or NULL. Kernels OR DS_DEV_ERR_* bits into
 *                it on input errors they detect; the affected cells get token
 *                -1 and logprob NaN. The caller clears it.
 *   stream       cudaStream_t.
 *
 * Noise: Gumbel G = -log(-log U) with U = ((x >> 8) + 1/2) 2^-24 and x word
 * (id & 3) of Philox4x32-10(counter = (id >> 2, t, request_id, iteration << 8
 * | row), key = (seed low, seed high)), t the request-local position.
 * The token maximises z[id] + tau * G[id] over the kept set.
 * Logits must be finite or -inf (no NaN, no +inf).
 *
 * Returns DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED (V > DS_MAX_VOCAB,
 * B beyond int32 cell counts) or DS_ERR_CUDA (launch failure).
 */
ds_status ds_sample(const int32_t* request_ids, const void* c_logits, const void* u_logits,
                    const int32_t* seq_lens, int32_t B, int32_t C, int32_t P, int32_t V,
                    const float* guidance, const float* temperature, float top_ratio,
                    uint64_t seed, uint32_t iteration, int32_t* out_tokens, float* out_logprobs,
                    uint32_t* d_status, void* stream);

/*
 * ds_sample_ex -- ds_sample with a kept fraction and an iteration per request.
 *
 * Defined by: "Add a sampler resource for discrete diffusion" (mstar PR #290),
 * Contract, which names the iterations of sample(...) in the plural, and the
 * per-request configuration of "Sampler support for discrete diffusion",
 * Hert4's first comment (guidance, temperature and the top-ratio filter are
 * per-request settings).
 *
 * Arguments as for ds_sample, plus:
 *   top_ratios   device float [B] or NULL. When given, request r keeps
 *                k_r = ceilf(top_ratios[r] * V) (fp32 product, clamped to
 *                [1, V]) and top_ratio is ignored; a ratio outside (0, 1]
 *                makes that request's cells token -1 / logprob NaN and sets
 *                DS_DEV_ERR_PARAM.
 *   iterations   device uint32 [B] or NULL. When given, request r's noise uses
 *                iterations[r] (< 2^24, else as an invalid ratio) and iteration
 *                is ignored.
 *   flags        OR of:
 *                DS_FLAG_KEEP_TIES: the kept set becomes every id whose z
 *                reaches the k-th largest z, so ids tied with the k-th are kept
 *                too (the pages keep the ceil(0.1 V) largest logits but do not
 *                say which of several tied at the cut; by default exactly k are
 *                kept, smallest ids first).
 *                DS_FLAG_SKIP_EXACT_PASS (diagnostic): the fast pass runs alone;
 *                a cell it cannot settle exactly is left with token
 *                DS_MARKED_TOKEN and an unspecified logprob instead of being
 *                finished by the exact pass that normally follows it on the
 *                stream. Every other cell is as without the flag. This lets a
 *                caller (a test, a profiler) count how often the exact pass runs.
 * With both arrays NULL and flags 0 this is ds_sample. Per-request arrays must
 * be 4-byte aligned. Unknown flag bits: DS_ERR_INVALID_ARG. Returns as ds_sample.
 */
#define DS_FLAG_KEEP_TIES 1u
#define DS_FLAG_SKIP_EXACT_PASS 2u
#define DS_MARKED_TOKEN (-2)
ds_status ds_sample_ex(const int32_t* request_ids, const void* c_logits, const void* u_logits,
                       const int32_t* seq_lens, int32_t B, int32_t C, int32_t P, int32_t V,
                       const float* guidance, const float* temperature, const float* top_ratios,
                       float top_ratio, uint64_t seed, const uint32_t* iterations, uint32_t iteration,
                       uint32_t flags, int32_t* out_tokens, float* out_logprobs, uint32_t* d_status,
                       void* stream);

/*
 * ds_greedy_lse -- per-row max, logsumexp and argmax of bf16 logits [n][V].
 *
 * Defined by: "perf: avoid full-vocab all-gather for draft greedy sampling"
 * (LightLLM PR #1517), Design and invariants: each vocabulary shard yields
 * its local max, log-sum-exp and argmax; ties go to the smallest token ID;
 * the selected token's exact probability is exp(selected_logit -
 * full_vocab_logsumexp), i.e. exp(out_max - out_lse) here. Inputs are not
 * rewritten: the id and the normaliser are returned beside the logits.
 *
 * Arguments:
 *   logits      device bf16 [n][V], V contiguous, 2-byte alignment.
 *   n, V        n >= 0 (0: nothing launched), V >= 1.
 *   out_max     device float [n]: max logit (exact).
 *   out_lse     device float [n]: logsumexp over the row (fp32 accumulation).
 *   out_argmax  device int32 [n]: smallest id attaining the max.
 *   stream      cudaStream_t.
 * Returns DS_OK, DS_ERR_INVALID_ARG or DS_ERR_CUDA.
 */
ds_status ds_greedy_lse(const void* logits, int32_t n, int32_t V, float* out_max, float* out_lse,
                        int32_t* out_argmax, void* stream);

/*
 * ds_merge_triples -- merge per-shard (max, lse, argmax) triples of a
 * vocabulary-sharded row into the full-row triple.
 *
 * Defined by: "perf: avoid full-vocab all-gather for draft greedy sampling"
 * (LightLLM PR #1517), Design and invariants: each rank holding a vocab shard
 * sends three FP32 words per token -- its local max, its local log-sum-exp and
 * its argmax as a global token id with the integer's bits kept in an FP32
 * word -- and the merge takes the global max, the token of the shard holding
 * it (the smallest global id when shards tie), and
 * lse = m + log(sum over shards of exp(lse_s - m)).
 *
 * Arguments:
 *   triples     device float [n][shards][3]: (max, lse, global argmax bits) per
 *               token and shard, shard order arbitrary. A shard whose logits
 *               are all -inf carries max = lse = -inf.
 *   n, shards   n >= 0 (0: nothing launched), shards >= 1.
 *   out_max     device float [n]: the largest shard max (exact).
 *   out_lse     device float [n]: the merged logsumexp (fp32, accurate expf/logf).
 *   out_argmax  device int32 [n]: the winner's global id; smallest id on ties.
 *   stream      cudaStream_t.
 * Returns DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED (n * shards * 3 > 2^40)
 * or DS_ERR_CUDA.
 */
ds_status ds_merge_triples(const float* triples, int32_t n, int32_t shards, float* out_max, float* out_lse,
                           int32_t* out_argmax, void* stream);

/* Output element types of ds_log_softmax. */
#define DS_DTYPE_F32 0
#define DS_DTYPE_BF16 1

/*
 * ds_log_softmax -- the greedy triple of every row plus the dense
 * log-softmax of bf16 logits [n][V].
 *
 * Defined by: the dense fallback path of "perf: avoid full-vocab all-gather
 * for draft greedy sampling" (LightLLM PR #1517), Design and invariants, for
 * callers that still need full log-probabilities: out[r][i] = x[r][i] -
 * logsumexp(x[r]). A row of up to about 262k logits is held in the shared
 * memory of a thread-block cluster, so the logits are read once and 4 (fp32)
 * or 2 (bf16) bytes per element are written. A longer row runs ds_greedy_lse
 * and then a pass that re-reads the logits. The triple equals ds_greedy_lse's
 * in max and argmax; lse agrees with it to fp32 rounding (the sums are taken
 * in another order).
 *
 * Arguments:
 *   logits      device bf16 [n][V], V contiguous, 2-byte alignment.
 *   n, V        n >= 0 (0: nothing launched), V >= 1.
 *   out         device [n][V] of out_dtype: fp32 (4-byte aligned) or bf16
 *               rounded to nearest even (2-byte aligned). A row of all -inf
 *               logits yields NaN (its logsumexp is -inf).
 *   out_dtype   DS_DTYPE_F32 or DS_DTYPE_BF16.
 *   out_max, out_lse, out_argmax  as for ds_greedy_lse.
 *   stream      cudaStream_t.
 * Returns DS_OK, DS_ERR_INVALID_ARG or DS_ERR_CUDA.
 */
ds_status ds_log_softmax(const void* logits, int32_t n, int32_t V, void* out, int32_t out_dtype, float* out_max,
                         float* out_lse, int32_t* out_argmax, void* stream);

/*
 * ds_reveal -- confidence ranking and reveal of one diffusion step.
 *
 * Defined by: "Sampler support for discrete diffusion" (mstar issue #267),
 * Hert4's first comment: after every cell is sampled, the caller ranks the
 * cells of a request's flattened [C, T] canvas by a confidence score and
 * commits only the top reveal_count (torch.topk over the flattened scores,
 * then a scatter). Here the order is score descending, then the flattened
 * index f = c * T_r + t ascending (the smallest index wins a tie, as the
 * greedy page's tie rule does for token ids), so exactly
 * min(reveal_counts[r], C * T_r) cells of request r are committed.
 *
 * Arguments (B requests, C rows, P = sum of seq_lens positions, packed as in
 * ds_sample):
 *   scores         device float [C][P]: the ranking score of every cell (for
 *                  example ds_sample's logprob, or the caller's own confidence
 *                  with its penalties applied). Not NaN; -0 and +0 tie.
 *   tokens         device int32 [C][P]: the sampled token of every cell.
 *   seq_lens       device int32 [B] (>= 0; sum == P).
 *   reveal_counts  device int32 [B]: cells to commit per request; <= 0 commits
 *                  none, >= C * T_r commits all.
 *   canvas         device int32 [C][P], in/out: committed cells get their
 *                  token; every other cell keeps its value.
 *   revealed       device uint8 [C][P] or NULL: 1 for the cells this call
 *                  committed, 0 for the others.
 *   d_status       device uint32 or NULL: DS_DEV_ERR_LAYOUT when seq_lens is
 *                  negative somewhere or does not sum to P (nothing written).
 *   stream         cudaStream_t.
 * Returns DS_OK, DS_ERR_INVALID_ARG, DS_ERR_UNSUPPORTED (C * P >= 2^32) or
 * DS_ERR_CUDA.
 */
ds_status ds_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
                    const int32_t* reveal_counts, int32_t B, int32_t C, int32_t P, int32_t* canvas,
                    uint8_t* revealed, uint32_t* d_status, void* stream);

/* Static description of a status code. Never NULL. */
const char* ds_status_string(ds_status s);

/* Kept count used by ds_sample: ceilf(top_ratio * V) in fp32, clamped to [1, V];
 * 0 when the arguments are invalid. Host-only, no CUDA call. */
int32_t ds_top_k(float top_ratio, int32_t V);

/* Number of kernels the library has launched in this process so far (every
 * successful launch by any entry point adds one; a call may launch one to three
 * kernels depending on its sizes and the device). For accounting by callers such
 * as benchmarks. Host-only, thread-safe, no CUDA call. */
uint64_t ds_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DSAMPLE_H */
