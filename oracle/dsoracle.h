/*
 * dsoracle.h -- C API of the CPU oracle for the vocab-wide sampling pass.
 *
 * TEST INFRASTRUCTURE ONLY. This oracle is a plain, slow, single-threaded
 * restatement of what the sampling pass computes. Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the product path
 * never does. It shares no code, header, table or constant generator with the
 * CUDA library.
 *
 * Sources restated (page title, part of page):
 *  - "Sampler support for discrete diffusion" (mstar issue #267), Hert4's
 *    first comment: log-softmax, argmax and max log-prob per cell; logits
 *    [C, T, V] with T ragged across requests; classifier-free-guidance combine
 *    of two logit tensors; top-ratio filter keeping ceil(0.1 * V) tokens;
 *    Gumbel sampling; a (token, logprob) is returned for every position the
 *    sampler is given, and ranking is left to the caller.
 *  - "Add a sampler resource for discrete diffusion" (mstar PR #290),
 *    "Contract": sample(request_ids, c_logits, u_logits, seq_lens, iterations)
 *    over [rows, positions, vocab] packed across requests; per-request guidance
 *    and temperature; no unconditional document for guidance 0.
 *  - "perf: avoid full-vocab all-gather for draft greedy sampling" (LightLLM
 *    PR #1517), "Design and invariants": per-row max, log-sum-exp and argmax;
 *    ties to the smallest token ID; p = exp(selected_logit - logsumexp).
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11.
 */
#ifndef DSORACLE_H
#define DSORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Flags of dso_sample_cells_ex. */
#define DSO_KEEP_TIES 1u  /* keep every id whose z equals the k-th largest z (kept set may exceed k) */

/* Return codes. */
#define DSO_OK 0
#define DSO_ERR_ARG 1      /* bad sizes, pointers or scalars */
#define DSO_ERR_LAYOUT 2   /* sum(seq_lens) != P, or u missing where g != 0 */

/* Philox4x32-10 block: out = Philox(ctr, key), 10 rounds. */
void dso_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Uniform U in (0,1) from one 32-bit word: ((x >> 8) + 0.5) * 2^-24, exact in double. */
double dso_uniform(uint32_t x);

/* Standard Gumbel variate G = -log(-log(U)) from one 32-bit word, in double. */
double dso_gumbel(uint32_t x);

/* Exact bf16 -> fp32 decode of one 16-bit pattern. */
float dso_bf16_to_float(uint16_t h);

/* Guided logit z = fmaf(g, c - u, c) (the subtraction rounded to fp32 first);
 * z = c exactly when g == 0. */
float dso_cfg(float c, float u, float g);

/* Kept count k = ceilf(top_ratio * (float)V), product in fp32, clamped to [1, V]. */
int32_t dso_top_k(float top_ratio, int32_t V);

/*
 * Sampling oracle over a list of cells.
 *
 * Layout (row-major, V contiguous): c_logits bf16 [C][P][V]; u_logits bf16
 * [C][P_u][V] with P_u = sum of seq_lens over requests with guidance != 0,
 * packed in request order (NULL allowed when no request has g != 0).
 * Request r owns positions [off_r, off_r + seq_lens[r]) of P.
 * A cell is (row c, position p); its flat index is c * P + p.
 *
 * For each listed cell index cells[j] this writes:
 *   out_tokens[j]    sampled token (argmax when the request's temperature is 0)
 *   out_logprobs[j]  z_tok - logsumexp(z), double
 *   out_lse[j]       logsumexp(z) over the full vocabulary, double   (nullable)
 *   out_max[j]       max z (fp32 value)                               (nullable)
 *   out_argmax[j]    smallest id attaining max z                      (nullable)
 *   out_top1[j], out_top2[j]  best and second-best perturbed score over the
 *                    kept set (double; -inf when absent; equal to max z /
 *                    -inf for temperature 0)                           (nullable)
 *   out_thresh_ties[j] number of ids tied with the k-th largest z that were
 *                    left out of the kept set (0 when the cut is clean) (nullable)
 * Returns DSO_OK or an error code (outputs untouched on error).
 */
int dso_sample_cells(const int32_t* request_ids, const uint16_t* c_logits,
                     const uint16_t* u_logits, const int32_t* seq_lens,
                     int32_t B, int32_t C, int32_t P, int32_t V,
                     const float* guidance, const float* temperature,
                     float top_ratio, uint64_t seed, uint32_t iteration,
                     const int64_t* cells, int64_t n_cells,
                     int32_t* out_tokens, double* out_logprobs,
                     double* out_lse, float* out_max, int32_t* out_argmax,
                     double* out_top1, double* out_top2,
                     int32_t* out_thresh_ties);

/*
 * As dso_sample_cells, with a kept fraction and an iteration per request:
 * request r uses top_ratios[r] (when top_ratios is not NULL, else top_ratio)
 * and iterations[r] (when iterations is not NULL, else iteration). The
 * contract's sample(..., iterations) names iterations in the plural ("Add a
 * sampler resource for discrete diffusion", Contract); each request's k is
 * ceilf(ratio_r * V) as for the scalar. flags: 0, or DSO_KEEP_TIES, which keeps
 * every id whose z equals the k-th largest z instead of exactly k ids (a filter
 * mode the pages leave open: "keep the ceil(0.1 V) largest" says nothing of
 * ties at the cut).
 */
int dso_sample_cells_ex(const int32_t* request_ids, const uint16_t* c_logits,
                        const uint16_t* u_logits, const int32_t* seq_lens,
                        int32_t B, int32_t C, int32_t P, int32_t V,
                        const float* guidance, const float* temperature,
                        const float* top_ratios, float top_ratio, uint64_t seed,
                        const uint32_t* iterations, uint32_t iteration, uint32_t flags,
                        const int64_t* cells, int64_t n_cells,
                        int32_t* out_tokens, double* out_logprobs,
                        double* out_lse, float* out_max, int32_t* out_argmax,
                        double* out_top1, double* out_top2,
                        int32_t* out_thresh_ties);

/*
 * Greedy oracle over a list of rows of logits bf16 [n][V]: per listed row,
 * max (fp32), logsumexp (double) and argmax (smallest id on ties).
 */
int dso_greedy_rows(const uint16_t* logits, int32_t n, int32_t V,
                    const int64_t* rows, int64_t n_rows,
                    float* out_max, double* out_lse, int32_t* out_argmax);

/*
 * Merge of per-shard (max, lse, argmax) triples for one token, as in the
 * vocab-sharded greedy path: the global max, the global logsumexp and the
 * winner's global id (ties to the smallest global id). Shard s covers global
 * ids [shard_base[s], ...). Argmax values are shard-local ids.
 */
void dso_merge_triples(const float* maxes, const double* lses, const int32_t* local_argmax,
                       const int32_t* shard_base, int32_t n_shards,
                       float* out_max, double* out_lse, int32_t* out_argmax);

/*
 * Confidence ranking and reveal of one diffusion step, as the caller does it
 * after sampling ("Sampler support for discrete diffusion", Hert4's first
 * comment: rank the cells of the flattened canvas by score and commit the top
 * reveal_count). Per request r (positions [off_r, off_r + T_r) of every row
 * c), the cells are flattened as f = c * T_r + t; the min(reveal_counts[r],
 * C * T_r) cells first in the order (score desc, f asc) get
 * canvas[c][off_r + t] = tokens[c][off_r + t] and revealed = 1; every other
 * cell of the request keeps its canvas value and gets revealed = 0. A
 * negative reveal count reveals nothing. revealed may be NULL.
 */
int dso_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
               const int32_t* reveal_counts, int32_t B, int32_t C, int32_t P,
               int32_t* canvas, uint8_t* revealed);

#ifdef __cplusplus
}
#endif

#endif /* DSORACLE_H */
