// dsoracle.cpp -- plain single-threaded CPU oracle of the vocab-wide sampling pass.
//
// TEST INFRASTRUCTURE ONLY: the CUDA library never includes, links or calls
// this file; only the tests, the smoke check and the benchmark's CPU-baseline
// leg load it. It is written to be checked by eye against the pages it
// restates, not to be fast: every step follows the definition in the order the
// pages give it, in double precision wherever the pages do not fix one.
// Build with -ffp-contract=off so that no a*b+c is silently fused.
//
// Parity pins: every function here is pinned by a CPU test under tests/
// (brute force, closed forms, library routines or cross-implementation checks);
// none is "parity unpinned".

#include "dsoracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

namespace {

// --- Philox4x32-10 (Salmon et al., SC'11, section 3.3 and table 2) ---------
// Round function on a 4x32 counter with a 2x32 key: two 32x32->64 products of
// the multipliers with counter words 0 and 2; the high halves are xored with
// the other counter words and the round key, the low halves are carried over.
// The key is bumped by the Weyl constants between rounds.
const uint32_t kPhiloxM0 = 0xD2511F53u;
const uint32_t kPhiloxM1 = 0xCD9E8D57u;
const uint32_t kPhiloxW0 = 0x9E3779B9u;  // golden ratio
const uint32_t kPhiloxW1 = 0xBB67AE85u;  // sqrt(3) - 1

void philox_round(uint32_t x[4], const uint32_t k[2]) {
  const uint64_t p0 = (uint64_t)kPhiloxM0 * (uint64_t)x[0];
  const uint64_t p1 = (uint64_t)kPhiloxM1 * (uint64_t)x[2];
  const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  const uint32_t y0 = hi1 ^ x[1] ^ k[0];
  const uint32_t y1 = lo1;
  const uint32_t y2 = hi0 ^ x[3] ^ k[1];
  const uint32_t y3 = lo0;
  x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
}

// Per-cell request lookup by a linear walk over seq_lens (plain, O(B)).
struct CellRequest {
  int32_t r;      // request index
  int32_t t;      // position local to the request
  int64_t u_pos;  // position of this cell's row inside u's packed positions (-1 if g == 0)
};

}  // namespace

extern "C" {

void dso_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k[2] = {key[0], key[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += kPhiloxW0;
      k[1] += kPhiloxW1;
    }
    philox_round(x, k);
  }
  out[0] = x[0]; out[1] = x[1]; out[2] = x[2]; out[3] = x[3];
}

double dso_uniform(uint32_t x) {
  // 24 random bits plus one half: the lattice midpoint, never 0 and never 1.
  return ((double)(x >> 8) + 0.5) * std::ldexp(1.0, -24);
}

double dso_gumbel(uint32_t x) {
  const double u = dso_uniform(x);
  return -std::log(-std::log(u));
}

float dso_bf16_to_float(uint16_t h) {
  // bf16 is the upper half of an IEEE binary32 pattern.
  const uint32_t bits = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &bits, sizeof f);
  return f;
}

float dso_cfg(float c, float u, float g) {
  // z = c + g * (c - u): the difference is rounded to fp32, then one fused
  // multiply-add. Guidance 0 means no unconditional logits: z = c exactly.
  if (g == 0.0f) return c;
  const float d = c - u;
  return std::fmaf(g, d, c);
}

int32_t dso_top_k(float top_ratio, int32_t V) {
  // ceil(ratio * V) with the product taken in fp32.
  const float prod = top_ratio * (float)V;
  int64_t k = (int64_t)std::ceil(prod);
  if (k < 1) k = 1;
  if (k > V) k = V;
  return (int32_t)k;
}

int dso_sample_cells(const int32_t* request_ids, const uint16_t* c_logits,
                     const uint16_t* u_logits, const int32_t* seq_lens,
                     int32_t B, int32_t C, int32_t P, int32_t V,
                     const float* guidance, const float* temperature,
                     float top_ratio, uint64_t seed, uint32_t iteration,
                     const int64_t* cells, int64_t n_cells,
                     int32_t* out_tokens, double* out_logprobs,
                     double* out_lse, float* out_max, int32_t* out_argmax,
                     double* out_top1, double* out_top2,
                     int32_t* out_thresh_ties) {
  return dso_sample_cells_ex(request_ids, c_logits, u_logits, seq_lens, B, C, P, V, guidance, temperature,
                             nullptr, top_ratio, seed, nullptr, iteration, 0u, cells, n_cells, out_tokens,
                             out_logprobs, out_lse, out_max, out_argmax, out_top1, out_top2, out_thresh_ties);
}

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
                        int32_t* out_thresh_ties) {
  if (B < 0 || C < 0 || P < 0 || V <= 0 || n_cells < 0) return DSO_ERR_ARG;
  if ((flags & ~DSO_KEEP_TIES) != 0u) return DSO_ERR_ARG;
  const bool keep_ties = (flags & DSO_KEEP_TIES) != 0u;
  if (n_cells == 0) return DSO_OK;
  if (!request_ids || !c_logits || !seq_lens || !guidance || !temperature || !cells ||
      !out_tokens || !out_logprobs)
    return DSO_ERR_ARG;
  if (C > 256) return DSO_ERR_ARG;
  // per-request kept fraction and iteration (the scalars when no array is given)
  for (int32_t r = 0; r < B; ++r) {
    const float ratio = top_ratios ? top_ratios[r] : top_ratio;
    const uint32_t it = iterations ? iterations[r] : iteration;
    if (!(ratio > 0.0f && ratio <= 1.0f)) return DSO_ERR_ARG;
    if (it >= (1u << 24)) return DSO_ERR_ARG;
  }

  // Packing: request r owns positions [off_r, off_r + T_r); u holds only the
  // requests with guidance != 0, in request order.
  int64_t total = 0, total_u = 0;
  for (int32_t r = 0; r < B; ++r) {
    if (seq_lens[r] < 0) return DSO_ERR_LAYOUT;
    total += seq_lens[r];
    if (guidance[r] != 0.0f) total_u += seq_lens[r];
  }
  if (total != P) return DSO_ERR_LAYOUT;
  if (total_u > 0 && u_logits == nullptr) return DSO_ERR_LAYOUT;
  const int64_t P_u = total_u;
  const uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  const double ninf = -std::numeric_limits<double>::infinity();

  std::vector<float> z((size_t)V);
  std::vector<int32_t> order((size_t)V);

  for (int64_t j = 0; j < n_cells; ++j) {
    const int64_t cell = cells[j];
    if (cell < 0 || cell >= (int64_t)C * P) return DSO_ERR_ARG;
    const int32_t c = (int32_t)(cell / P);
    const int32_t p = (int32_t)(cell % P);

    // Request lookup.
    CellRequest req{-1, 0, -1};
    int64_t off = 0, off_u = 0;
    for (int32_t r = 0; r < B; ++r) {
      if (p < off + seq_lens[r]) {
        req.r = r;
        req.t = (int32_t)(p - off);
        req.u_pos = (guidance[r] != 0.0f) ? off_u + req.t : -1;
        break;
      }
      off += seq_lens[r];
      if (guidance[r] != 0.0f) off_u += seq_lens[r];
    }
    if (req.r < 0) return DSO_ERR_LAYOUT;
    const float g = guidance[req.r];
    const float tau = temperature[req.r];
    if (!(tau >= 0.0f) || std::isnan(g)) return DSO_ERR_ARG;
    const int32_t k = dso_top_k(top_ratios ? top_ratios[req.r] : top_ratio, V);
    const uint32_t iteration_r = iterations ? iterations[req.r] : iteration;

    // Step 1: guided logits z over the full vocabulary.
    const uint16_t* crow = c_logits + ((int64_t)c * P + p) * (int64_t)V;
    const uint16_t* urow = (req.u_pos >= 0) ? u_logits + ((int64_t)c * P_u + req.u_pos) * (int64_t)V : nullptr;
    for (int32_t i = 0; i < V; ++i) {
      const float cf = dso_bf16_to_float(crow[i]);
      const float uf = urow ? dso_bf16_to_float(urow[i]) : 0.0f;
      z[(size_t)i] = dso_cfg(cf, uf, g);
    }

    // Step 2: max, smallest id attaining it, and logsumexp in double.
    float m = z[0];
    int32_t a = 0;
    for (int32_t i = 1; i < V; ++i) {
      if (z[(size_t)i] > m) {
        m = z[(size_t)i];
        a = i;
      }
    }
    double lse;
    if (m == -std::numeric_limits<float>::infinity()) {
      lse = ninf;
    } else {
      double s = 0.0;
      for (int32_t i = 0; i < V; ++i) s += std::exp((double)z[(size_t)i] - (double)m);
      lse = (double)m + std::log(s);
    }

    int32_t token;
    double top1, top2;
    int32_t thresh_ties = 0;
    if (tau == 0.0f) {
      // Temperature 0: the argmax, no filter and no noise.
      token = a;
      top1 = (double)m;
      top2 = ninf;
    } else {
      // Step 3: the k largest z, ties broken toward the smallest id.
      for (int32_t i = 0; i < V; ++i) order[(size_t)i] = i;
      auto before = [&](int32_t x, int32_t y) {
        if (z[(size_t)x] != z[(size_t)y]) return z[(size_t)x] > z[(size_t)y];
        return x < y;
      };
      if (k < V) std::nth_element(order.begin(), order.begin() + (k - 1), order.end(), before);
      // The k-th element of the order sits at position k-1; count ids equal in z to it
      // that fall outside the kept set (diagnostic only). With keep_ties they are
      // kept: the kept set grows to every id whose z reaches the k-th largest z.
      int32_t n_kept = k;
      if (k < V) {
        const float zk = z[(size_t)order[(size_t)(k - 1)]];
        for (int32_t q = k; q < V; ++q)
          if (z[(size_t)order[(size_t)q]] == zk) {
            if (keep_ties)
              std::swap(order[(size_t)n_kept++], order[(size_t)q]);
            else
              ++thresh_ties;
          }
      }
      // Step 4: Gumbel-max over the kept set at temperature tau.
      int32_t best = -1;
      top1 = ninf;
      top2 = ninf;
      for (int32_t q = 0; q < n_kept; ++q) {
        const int32_t i = order[(size_t)q];
        const uint32_t ctr[4] = {(uint32_t)i >> 2, (uint32_t)req.t, (uint32_t)request_ids[req.r],
                                 (iteration_r << 8) | (uint32_t)c};
        uint32_t words[4];
        dso_philox4x32_10(ctr, key, words);
        const double G = dso_gumbel(words[i & 3]);
        const double score = (double)z[(size_t)i] + (double)tau * G;
        if (best < 0 || score > top1 || (score == top1 && i < best)) {
          top2 = top1;
          top1 = score;
          best = i;
        } else if (score > top2) {
          top2 = score;
        }
      }
      token = best;
    }

    out_tokens[j] = token;
    out_logprobs[j] = (double)z[(size_t)token] - lse;
    if (out_lse) out_lse[j] = lse;
    if (out_max) out_max[j] = m;
    if (out_argmax) out_argmax[j] = a;
    if (out_top1) out_top1[j] = top1;
    if (out_top2) out_top2[j] = top2;
    if (out_thresh_ties) out_thresh_ties[j] = thresh_ties;
  }
  return DSO_OK;
}

int dso_greedy_rows(const uint16_t* logits, int32_t n, int32_t V,
                    const int64_t* rows, int64_t n_rows,
                    float* out_max, double* out_lse, int32_t* out_argmax) {
  if (n < 0 || V <= 0 || n_rows < 0) return DSO_ERR_ARG;
  if (n_rows == 0) return DSO_OK;
  if (!logits || !rows || !out_max || !out_lse || !out_argmax) return DSO_ERR_ARG;
  for (int64_t j = 0; j < n_rows; ++j) {
    const int64_t row = rows[j];
    if (row < 0 || row >= n) return DSO_ERR_ARG;
    const uint16_t* x = logits + row * (int64_t)V;
    float m = dso_bf16_to_float(x[0]);
    int32_t a = 0;
    for (int32_t i = 1; i < V; ++i) {
      const float v = dso_bf16_to_float(x[i]);
      if (v > m) {
        m = v;
        a = i;
      }
    }
    double lse;
    if (m == -std::numeric_limits<float>::infinity()) {
      lse = -std::numeric_limits<double>::infinity();
    } else {
      double s = 0.0;
      for (int32_t i = 0; i < V; ++i) s += std::exp((double)dso_bf16_to_float(x[i]) - (double)m);
      lse = (double)m + std::log(s);
    }
    out_max[j] = m;
    out_lse[j] = lse;
    out_argmax[j] = a;
  }
  return DSO_OK;
}

void dso_merge_triples(const float* maxes, const double* lses, const int32_t* local_argmax,
                       const int32_t* shard_base, int32_t n_shards,
                       float* out_max, double* out_lse, int32_t* out_argmax) {
  // Global max; the winner is the shard holding it, smallest global id on ties.
  float m = -std::numeric_limits<float>::infinity();
  int32_t a = -1;
  for (int32_t s = 0; s < n_shards; ++s) {
    const int32_t gid = shard_base[s] + local_argmax[s];
    if (a < 0 || maxes[s] > m || (maxes[s] == m && gid < a)) {
      m = maxes[s];
      a = gid;
    }
  }
  // Global logsumexp from the shard logsumexps: log sum_s exp(lse_s).
  double lse;
  if (m == -std::numeric_limits<float>::infinity()) {
    lse = -std::numeric_limits<double>::infinity();
  } else {
    double acc = 0.0;
    for (int32_t s = 0; s < n_shards; ++s) acc += std::exp(lses[s] - (double)m);
    lse = (double)m + std::log(acc);
  }
  *out_max = m;
  *out_lse = lse;
  *out_argmax = a;
}

int dso_reveal(const float* scores, const int32_t* tokens, const int32_t* seq_lens,
               const int32_t* reveal_counts, int32_t B, int32_t C, int32_t P,
               int32_t* canvas, uint8_t* revealed) {
  if (B < 0 || C < 0 || P < 0) return DSO_ERR_ARG;
  int64_t off = 0;
  for (int32_t r = 0; r < B; ++r) off += seq_lens[r] < 0 ? 0 : seq_lens[r];
  if (off != P) return DSO_ERR_LAYOUT;
  off = 0;
  for (int32_t r = 0; r < B; ++r) {
    const int64_t T = seq_lens[r] < 0 ? 0 : seq_lens[r];
    const int64_t n = (int64_t)C * T;
    // the request's cells in rank order: higher score first, then lower flattened index
    std::vector<int64_t> f(n);
    for (int64_t i = 0; i < n; ++i) f[i] = i;
    auto score_of = [&](int64_t fi) {
      const int64_t c = fi / (T > 0 ? T : 1), t = fi - c * T;
      return scores[c * (int64_t)P + off + t];
    };
    std::sort(f.begin(), f.end(), [&](int64_t a, int64_t b) {
      const float sa = score_of(a), sb = score_of(b);
      if (sa != sb) return sa > sb;
      return a < b;
    });
    int64_t k = reveal_counts[r];
    if (k < 0) k = 0;
    if (k > n) k = n;
    for (int64_t i = 0; i < n; ++i) {
      const int64_t fi = f[i];
      const int64_t c = fi / T, t = fi - c * T;
      const int64_t cell = c * (int64_t)P + off + t;
      if (i < k) canvas[cell] = tokens[cell];
      if (revealed) revealed[cell] = (uint8_t)(i < k ? 1 : 0);
    }
    off += T;
  }
  return DSO_OK;
}

}  // extern "C"
