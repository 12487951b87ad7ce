/*
 * Oracle: the verify-and-sample step, written out plainly.
 * TEST INFRASTRUCTURE ONLY (see orc.h for the sources, the precision rule and
 * what a "margin" is).
 *
 * Conventions shared by every function here:
 *  - Row (b, j) of a [B, R, V] tensor is flat row b*R + j; rows are ld elements apart.
 *  - Temperatures below ORC_GREEDY_T (and NaN) mean greedy: one-hot at the argmax.
 *  - top_k <= 0 or >= V means no top-k; top_p >= 1 means no top-p.
 *  - "Order" is value descending, then token id ascending (the argmax keeps the
 *    lowest id on ties; top-k keeps exactly k, lowest ids first among equals).
 *  - A token id outside [0, V) is never accepted and has probability 0.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "orc.h"

static int is_greedy(float T) { return !(T >= ORC_GREEDY_T); }

/* Argmax with the lowest index on ties (greedy_argmax: same tokens as torch.argmax). */
int64_t orc_argmax(const float* x, int64_t V) {
  int64_t best = 0;
  for (int64_t i = 1; i < V; ++i)
    if (x[i] > x[best]) best = i;
  return best;
}

typedef struct {
  float v;
  int64_t i;
} orc_item;

static int cmp_order(const void* a, const void* b) {
  const orc_item* x = (const orc_item*)a;
  const orc_item* y = (const orc_item*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i ? 1 : 0);
}

static double dmin(double a, double b) { return a < b ? a : b; }

/*
 * The filtered distribution of one row, p''.
 *
 *  1. Temperature softmax (flashinfer.py verify(): softmax(logits, temperature)):
 *     p_i = exp((l_i - M)/T) / sum_k exp((l_k - M)/T), M the row maximum.
 *     Greedy temperatures give the one-hot vector at the argmax.
 *     For a row of probabilities (is_logits == 0) the weights are the values.
 *  2. Top-k renorm: keep the first k tokens in order, renormalise.
 *  3. Top-p renorm on the top-k result (the fused kernel replaces back-to-back
 *     top_k_renorm_prob and top_p_renorm_prob): walking the kept tokens in
 *     order, keep the token at rank r iff r == 0 or the mass strictly before it
 *     is below top_p times the kept mass; renormalise.
 *
 * Returns the top-p margin: the distance, relative to the kept mass, between
 * the cut and top_p at the two comparisons that fixed the cut (+inf if no cut
 * or the row is greedy). out receives p'' (0 outside the kept set).
 */
double orc_filter_row(const float* vals, int64_t V, int is_logits, float T,
                      int32_t top_k, float top_p, double* out, int64_t* argmax_out) {
  return orc_filter_row_ex(vals, V, is_logits, T, top_k, top_p, 0.0f, 0, out, argmax_out);
}

/*
 * orc_filter_row with the two variations of the single-step samplers:
 *
 *  joint (TokenSpeed sample(): top_k_top_p_sampling_from_probs with
 *  filter_apply_order="joint"): top-k and top-p are both measured on the
 *  unfiltered p. The top-p set is then the shortest prefix of the order whose mass
 *  reaches top_p times the whole row's mass, and the kept set is its intersection
 *  with the top-k prefix. With joint == 0 the nucleus is measured on the top-k
 *  renormalised p' (step 3 above). The two differ only when both knobs are active.
 *
 *  min_p (TensorRT-LLM fused_sample_from_logits(..., min_ps, ...)): of the tokens
 *  the two knobs keep, only those whose weight is at least min_p times the largest
 *  weight stay (min_p is clamped to [0, 1], so the argmax always stays). The test is
 *  a ratio of weights, so it reads the same before or after any renormalisation.
 *
 * The margin adds, for min_p, the log-ratio distance of the last kept and the first
 * dropped token from ln(min_p), over max(1, |ln min_p|).
 */
double orc_filter_row_ex(const float* vals, int64_t V, int is_logits, float T,
                         int32_t top_k, float top_p, float min_p, int joint, double* out,
                         int64_t* argmax_out) {
  int64_t am = orc_argmax(vals, V);
  if (argmax_out) *argmax_out = am;
  for (int64_t i = 0; i < V; ++i) out[i] = 0.0;
  if (is_logits && is_greedy(T)) {
    out[am] = 1.0;
    return INFINITY;
  }
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  orc_item* it = (orc_item*)malloc(sizeof(orc_item) * (size_t)V);
  double M = (double)vals[am];
  for (int64_t i = 0; i < V; ++i) {
    if (is_logits)
      w[i] = (vals[i] == -INFINITY) ? 0.0 : exp(((double)vals[i] - M) / (double)T);
    else
      w[i] = (double)vals[i];
    it[i].v = vals[i];
    it[i].i = i;
  }
  qsort(it, (size_t)V, sizeof(orc_item), cmp_order);

  int64_t nk = (top_k > 0 && (int64_t)top_k < V) ? (int64_t)top_k : V;
  double Zk = 0.0;
  for (int64_t r = 0; r < nk; ++r) Zk += w[it[r].i];
  /* the mass top_p is a fraction of: the top-k mass, or the whole row's (joint) */
  double Zref = Zk;
  if (joint) {
    Zref = 0.0;
    for (int64_t r = 0; r < V; ++r) Zref += w[it[r].i];
  }

  double margin = INFINITY;
  int64_t nkeep = nk;
  if (top_p < 1.0f) {
    double P = (double)top_p * Zref;
    double S = 0.0;
    int64_t r = 0;
    for (; r < nk; ++r) {
      if (r == 0 || S < P) {
        S += w[it[r].i];
      } else {
        break;
      }
    }
    nkeep = r;
    int64_t rl = nkeep - 1;
    double S_before = S - w[it[rl].i];
    if (rl > 0) margin = dmin(margin, fabs(P - S_before) / Zref);
    if (nkeep < nk) margin = dmin(margin, fabs(S - P) / Zref);
  }
  if (min_p > 0.0f) {
    double mp = min_p < 1.0f ? (double)min_p : 1.0;
    double w0 = w[it[0].i];
    double thr = mp * w0;
    int64_t r = 1;
    while (r < nkeep && w[it[r].i] >= thr) ++r;
    double lmp = log(mp), scale = fabs(lmp) > 1.0 ? fabs(lmp) : 1.0;
    if (r > 1) margin = dmin(margin, fabs(log(w[it[r - 1].i] / w0) - lmp) / scale);
    if (r < nkeep && w[it[r].i] > 0.0)
      margin = dmin(margin, fabs(log(w[it[r].i] / w0) - lmp) / scale);
    nkeep = r;
  }
  double Z = 0.0;
  for (int64_t r = 0; r < nkeep; ++r) Z += w[it[r].i];
  for (int64_t r = 0; r < nkeep; ++r) out[it[r].i] = w[it[r].i] / Z;
  free(w);
  free(it);
  return margin;
}

/* Chosen-token logprob from raw logits at temperature 1 (gather_token_logprobs_torch
 * is given the unprocessed logits): l_t - M - ln sum exp(l - M). */
static double logprob_from_logits(const float* x, int64_t V, int64_t t) {
  int64_t am = orc_argmax(x, V);
  double M = (double)x[am];
  double s = 0.0;
  for (int64_t i = 0; i < V; ++i)
    if (x[i] != -INFINITY) s += exp((double)x[i] - M);
  return ((double)x[t] - M) - log(s);
}

void orc_softmax_temp(const float* logits, int64_t rows, int64_t V, int64_t ld,
                      const float* temperature, double* probs_out) {
  for (int64_t r = 0; r < rows; ++r) {
    float T = temperature ? temperature[r] : 1.0f;
    orc_filter_row(logits + r * ld, V, 1, T, 0, 1.0f, probs_out + r * V, NULL);
  }
}

void orc_topk_topp_renorm(const float* probs, int64_t rows, int64_t V, int64_t ld,
                          const int32_t* top_k, const float* top_p, double* out,
                          double* margin_out) {
  for (int64_t r = 0; r < rows; ++r) {
    int32_t k = top_k ? top_k[r] : 0;
    float p = top_p ? top_p[r] : 1.0f;
    double m = orc_filter_row(probs + r * ld, V, 0, 1.0f, k, p, out + r * V, NULL);
    if (margin_out) margin_out[r] = m;
  }
}

/* Greedy chain verification (verify_chain_greedy on the target argmax): draft j is
 * accepted while it equals the argmax of target row j; the argmax of the first
 * mismatching row (or of row D, the bonus) follows; then -1. accept_length counts
 * the emitted tokens, accept_index holds their flat positions b*(D+1)+j. */
void orc_verify_chain_greedy(const float* logits, int64_t B, int32_t D, int64_t V,
                             int64_t ld, const int32_t* draft_tokens,
                             int32_t* accepted_tokens, int32_t* accept_length,
                             int32_t* accept_index, double* logprobs) {
  const int64_t R = (int64_t)D + 1;
  for (int64_t b = 0; b < B; ++b) {
    int32_t js = D;
    for (int32_t j = 0; j < D; ++j) {
      int64_t a = orc_argmax(logits + (b * R + j) * ld, V);
      if ((int64_t)draft_tokens[b * D + j] != a) {
        js = j;
        break;
      }
    }
    for (int64_t j = 0; j < R; ++j) {
      int32_t tok = -1;
      if (j < js) tok = draft_tokens[b * D + j];
      else if (j == js) tok = (int32_t)orc_argmax(logits + (b * R + j) * ld, V);
      accepted_tokens[b * R + j] = tok;
      if (accept_index) accept_index[b * R + j] = (j <= js) ? (int32_t)(b * R + j) : -1;
      if (logprobs)
        logprobs[b * R + j] =
            (j <= js) ? logprob_from_logits(logits + (b * R + j) * ld, V, tok) : 0.0;
    }
    accept_length[b] = js + 1;
  }
}

/*
 * Chain speculative sampling (rejection_sampling_one_model contract; the
 * target-only variant is chain_speculative_sampling_target_only with no draft probs).
 *
 * For draft position j = 0..D-1 with draft token x:
 *   with draft probs q:  accept iff u_j * q_j(x) < p_j(x)       (min(1, p/q) rule)
 *   target-only:         accept iff u_j < p_j(x)                (q is the point mass at x)
 * At the first rejection j*, draw from norm(max(p_j* - q_j*, 0)) (target-only: p_j*
 * with x zeroed); if all D are accepted, draw the bonus from p_D. The draw takes
 * coin u_D: the smallest token i whose inclusive prefix mass (token-id order)
 * exceeds u_D times the total. If the residual mass is zero, draw from p_j*.
 * p is the filtered distribution (temperature, top-k, top-p) when the target is
 * logits, and the given fp32 row when it is probabilities.
 *
 * margin_out[b] is the smallest margin of any floating-point decision the request
 * took (accept tests, top-p cuts of the rows it used, the final draw).
 */
void orc_chain_spec_sampling(const float* target, int target_is_logits, int64_t B,
                             int32_t D, int64_t V, int64_t ld,
                             const float* temperature, const int32_t* top_k,
                             const float* top_p, const float* draft_probs,
                             int64_t ld_draft, const int32_t* draft_tokens,
                             const int64_t* seed, const int64_t* offset,
                             const float* uniforms, int32_t* accepted_tokens,
                             int32_t* accept_length, int32_t* accept_index,
                             double* logprobs, double* margin_out) {
  orc_chain_spec_sampling_ex(target, target_is_logits, B, D, V, ld, temperature, top_k, top_p,
                             NULL, 1.0f, 1.0f, draft_probs, ld_draft, draft_tokens, seed, offset,
                             uniforms, accepted_tokens, accept_length, accept_index, logprobs,
                             margin_out);
}

/*
 * orc_chain_spec_sampling with min_p filtering of the target rows (logits only; see
 * orc_filter_row_ex) and relaxed acceptance (TokenSpeed verify() passes threshold_single
 * and threshold_acc to chain_speculative_sampling_target_only; the pages give no
 * formula, and this is the reading taken): in target-only mode draft x is accepted iff
 *     p(x) >= threshold_single   or   u * threshold_acc < p(x),
 * so thresholds of 1 give plain rejection sampling (u < p(x)) and smaller ones accept
 * more. A threshold outside (0, 1) means 1. With draft probabilities both must be 1.
 * The margin adds |u * threshold_acc - p(x)| and |p(x) - threshold_single| for each
 * relaxed test.
 */
void orc_chain_spec_sampling_ex(const float* target, int target_is_logits, int64_t B,
                                int32_t D, int64_t V, int64_t ld, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p,
                                float threshold_single, float threshold_acc,
                                const float* draft_probs, int64_t ld_draft,
                                const int32_t* draft_tokens, const int64_t* seed,
                                const int64_t* offset, const float* uniforms,
                                int32_t* accepted_tokens, int32_t* accept_length,
                                int32_t* accept_index, double* logprobs, double* margin_out) {
  const int64_t R = (int64_t)D + 1;
  const float ts = (threshold_single > 0.0f && threshold_single < 1.0f) ? threshold_single : 1.0f;
  const float ta = (threshold_acc > 0.0f && threshold_acc < 1.0f) ? threshold_acc : 1.0f;
  const int relaxed = (ts < 1.0f || ta < 1.0f) && !draft_probs;
  double* dist = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  float* u = (float*)malloc(sizeof(float) * (size_t)R);
  for (int64_t b = 0; b < B; ++b) {
    float T = temperature ? temperature[b] : 1.0f;
    int32_t k = top_k ? top_k[b] : 0;
    float p = top_p ? top_p[b] : 1.0f;
    float mp = min_p ? min_p[b] : 0.0f;
    int greedy_row = target_is_logits && is_greedy(T); /* p is one-hot at the argmax */
    for (int64_t j = 0; j < R; ++j)
      u[j] = uniforms ? uniforms[b * R + j]
                      : orc_verify_coin((uint64_t)seed[b], (uint64_t)offset[b], (uint32_t)j);
    double margin = INFINITY;
    int32_t js = D;
    for (int32_t j = 0; j < D; ++j) {
      const float* row = target + (b * R + j) * ld;
      int32_t x = draft_tokens[b * D + j];
      int valid = (x >= 0 && (int64_t)x < V);
      int acc;
      if (target_is_logits) {
        margin = dmin(margin, orc_filter_row_ex(row, V, 1, T, k, p, mp, 0, dist, NULL));
        double px = valid ? dist[x] : 0.0;
        int exact = greedy_row || px == 0.0; /* one-hot rows and unkept tokens */
        if (draft_probs) {
          double qx = valid ? (double)draft_probs[(b * D + j) * ld_draft + x] : 0.0;
          double lhs = (double)u[j] * qx;
          acc = lhs < px;
          if (!exact) margin = dmin(margin, fabs(lhs - px));
        } else if (relaxed) {
          double lhs = (double)u[j] * (double)ta;
          acc = px >= (double)ts || lhs < px;
          if (!exact) margin = dmin(margin, dmin(fabs(lhs - px), fabs(px - (double)ts)));
        } else {
          acc = (double)u[j] < px;
          if (!exact) margin = dmin(margin, fabs((double)u[j] - px));
        }
      } else {
        float pxf = valid ? row[x] : 0.0f;
        if (draft_probs) {
          float qxf = valid ? draft_probs[(b * D + j) * ld_draft + x] : 0.0f;
          volatile float prod = u[j] * qxf; /* one fp32 multiply, rounded to nearest */
          acc = prod < pxf;
        } else if (relaxed) {
          volatile float lhs = u[j] * ta; /* one fp32 multiply, rounded to nearest */
          acc = pxf >= ts || lhs < pxf;
        } else {
          acc = u[j] < pxf;
        }
      }
      if (!acc) {
        js = j;
        break;
      }
    }

    /* The final draw from row js. */
    const float* row = target + (b * R + js) * ld;
    if (target_is_logits) {
      double m = orc_filter_row_ex(row, V, 1, T, k, p, mp, 0, dist, NULL);
      if (js == D) margin = dmin(margin, m); /* rows < D were counted above */
    } else {
      for (int64_t i = 0; i < V; ++i) dist[i] = (double)row[i];
    }
    if (js < D) {
      int32_t x = draft_tokens[b * D + js];
      if (draft_probs) {
        const float* q = draft_probs + (b * D + js) * ld_draft;
        for (int64_t i = 0; i < V; ++i) {
          if (target_is_logits) {
            double d = dist[i] - (double)q[i];
            w[i] = d > 0.0 ? d : 0.0;
          } else {
            float d = row[i] - q[i]; /* elementwise in fp32, as the inputs are fp32 */
            w[i] = d > 0.0f ? (double)d : 0.0;
          }
        }
      } else {
        for (int64_t i = 0; i < V; ++i) w[i] = dist[i];
        if (x >= 0 && (int64_t)x < V) w[x] = 0.0;
      }
    } else {
      for (int64_t i = 0; i < V; ++i) w[i] = dist[i];
    }
    double Z = 0.0;
    for (int64_t i = 0; i < V; ++i) Z += w[i];
    if (!(Z > 0.0)) {
      for (int64_t i = 0; i < V; ++i) w[i] = dist[i];
      Z = 0.0;
      for (int64_t i = 0; i < V; ++i) Z += w[i];
      margin = 0.0; /* a degenerate residual is always reported */
    }
    /* A distribution with a single token of nonzero mass draws that token for
     * every coin, so such a draw is exact. */
    int64_t nnz = 0;
    for (int64_t i = 0; i < V; ++i) nnz += (w[i] > 0.0);
    int exact_draw = (nnz == 1);
    double t = (double)u[D] * Z;
    int64_t tok = -1, last_pos = -1;
    double S = 0.0;
    for (int64_t i = 0; i < V; ++i) {
      if (w[i] > 0.0) {
        last_pos = i;
        if (S + w[i] > t) {
          tok = i;
          if (!exact_draw) margin = dmin(margin, dmin(t - S, S + w[i] - t) / Z);
          break;
        }
        S += w[i];
      }
    }
    if (tok < 0) {
      tok = last_pos;
      margin = 0.0;
    }

    for (int64_t j = 0; j < R; ++j) {
      int32_t t_out = -1;
      if (j < js) t_out = draft_tokens[b * D + j];
      else if (j == js) t_out = (int32_t)tok;
      accepted_tokens[b * R + j] = t_out;
      if (accept_index) accept_index[b * R + j] = (j <= js) ? (int32_t)(b * R + j) : -1;
      if (logprobs) {
        double lp = 0.0;
        const float* rj = target + (b * R + j) * ld;
        if (j <= js && t_out >= 0 && (int64_t)t_out < V)
          lp = target_is_logits ? logprob_from_logits(rj, V, t_out) : log((double)rj[t_out]);
        logprobs[b * R + j] = lp;
      }
    }
    accept_length[b] = js + 1;
    if (margin_out) margin_out[b] = margin;
  }
  free(dist);
  free(w);
  free(u);
}

/*
 * Ragged verification (TensorRT-LLM SpecMetadata.verify_lens / qo_indptr; ragged_helpers
 * scatter_ragged_to_padded, count_accepted_ragged, fill_padded_rows_onehot, and the
 * accept ceiling min(num_accepted, verify_lens)): request b owns the packed target rows
 * qo_indptr[b] .. qo_indptr[b+1] - 1, L_b of them, and verifies only its own window: its
 * first D_b = L_b - 1 drafts, exactly as a request with D = D_b drafts (the pages pad the
 * rows to a rectangle, fill the padding rows one-hot and cap the count at L_b so that no
 * token past the window is committed; here the window is verified directly). Drafts,
 * draft probabilities and coins keep their padded layouts ([B, D], [B*D, ld_draft],
 * [B, D+1]: the final draw's coin is entry D_b), the outputs are padded to [B, D+1]
 * (-1, -1, 0 past the emitted tokens) and accept_index holds packed row numbers
 * qo_indptr[b] + j. A window outside [1, D+1] rows is left unverified (accept_length 0).
 */
static void ragged_pad(int64_t b, int32_t D, int32_t Db, int64_t first, const int32_t* acc,
                       int32_t alen, const int32_t* idx, const double* lp,
                       int32_t* accepted_tokens, int32_t* accept_length, int32_t* accept_index,
                       double* logprobs) {
  const int64_t R = (int64_t)D + 1;
  for (int64_t j = 0; j < R; ++j) {
    int in = j <= Db && alen > 0;
    accepted_tokens[b * R + j] = in ? acc[j] : -1;
    if (accept_index)
      accept_index[b * R + j] = (in && idx[j] >= 0) ? (int32_t)(first + idx[j]) : -1;
    if (logprobs) logprobs[b * R + j] = in ? lp[j] : 0.0;
  }
  accept_length[b] = alen;
}

void orc_verify_chain_greedy_ragged(const float* logits, int64_t B, int32_t D, int64_t V,
                                    int64_t ld, const int32_t* qo_indptr,
                                    const int32_t* draft_tokens, int32_t* accepted_tokens,
                                    int32_t* accept_length, int32_t* accept_index,
                                    double* logprobs) {
  int32_t acc[ORC_MAX_R], idx[ORC_MAX_R];
  double lp[ORC_MAX_R];
  for (int64_t b = 0; b < B; ++b) {
    const int64_t first = qo_indptr[b];
    const int64_t L = (int64_t)qo_indptr[b + 1] - first;
    int32_t alen = 0;
    if (L >= 1 && L <= (int64_t)D + 1) {
      const int32_t Db = (int32_t)L - 1;
      orc_verify_chain_greedy(logits + first * ld, 1, Db, V, ld, draft_tokens + b * D, acc,
                              &alen, idx, lp);
    }
    ragged_pad(b, D, (int32_t)L - 1, first, acc, alen, idx, lp, accepted_tokens, accept_length,
               accept_index, logprobs);
  }
}

void orc_chain_spec_sampling_ragged(const float* target, int target_is_logits, int64_t B,
                                    int32_t D, int64_t V, int64_t ld, const int32_t* qo_indptr,
                                    const float* temperature, const int32_t* top_k,
                                    const float* top_p, const float* min_p,
                                    float threshold_single, float threshold_acc,
                                    const float* draft_probs, int64_t ld_draft,
                                    const int32_t* draft_tokens, const int64_t* seed,
                                    const int64_t* offset, const float* uniforms,
                                    int32_t* accepted_tokens, int32_t* accept_length,
                                    int32_t* accept_index, double* logprobs,
                                    double* margin_out) {
  int32_t acc[ORC_MAX_R], idx[ORC_MAX_R];
  double lp[ORC_MAX_R];
  for (int64_t b = 0; b < B; ++b) {
    const int64_t first = qo_indptr[b];
    const int64_t L = (int64_t)qo_indptr[b + 1] - first;
    int32_t alen = 0;
    double m = INFINITY;
    if (L >= 1 && L <= (int64_t)D + 1) {
      const int32_t Db = (int32_t)L - 1;
      orc_chain_spec_sampling_ex(
          target + first * ld, target_is_logits, 1, Db, V, ld,
          temperature ? temperature + b : NULL, top_k ? top_k + b : NULL,
          top_p ? top_p + b : NULL, min_p ? min_p + b : NULL, threshold_single, threshold_acc,
          draft_probs ? draft_probs + b * D * ld_draft : NULL, ld_draft, draft_tokens + b * D,
          seed ? seed + b : NULL, offset ? offset + b : NULL,
          uniforms ? uniforms + b * ((int64_t)D + 1) : NULL, acc, &alen, idx, lp, &m);
    }
    ragged_pad(b, D, (int32_t)L - 1, first, acc, alen, idx, lp, accepted_tokens, accept_length,
               accept_index, logprobs);
    if (margin_out) margin_out[b] = m;
  }
}

/*
 * Single-step sampling from logits (TokenSpeed sample(): softmax with temperature,
 * then top_k_top_p_sampling_from_probs(..., filter_apply_order="joint", seed, offset);
 * TensorRT-LLM advanced_sample_draft / advanced_sample_draft_block:
 * fused_sample_from_logits_with_probs(logits, temperatures, top_ks, top_ps, min_ps, seed,
 * offset), whose probabilities are stored for the next verify step).
 *
 * Row r = b * n_per_req + j (knobs per row, seed and offset per request b) is filtered
 * by orc_filter_row_ex (joint or top-k-first order, min_p) and one token is drawn from
 * the kept distribution by the inverse CDF in token-id order: the smallest token whose
 * inclusive prefix mass exceeds u times the total, with the coin u of position j of the
 * request's verify stream (or uniforms[r]). A greedy row takes its argmax. probs_out
 * receives the kept distribution (0 outside it), logprobs_out the temperature-1
 * log-softmax of the chosen token, margin_out the smallest decision margin (filter cuts
 * and the draw).
 */
void orc_sample_from_logits(const float* logits, int64_t B, int32_t n_per_req, int64_t V,
                            int64_t ld, const float* temperature, const int32_t* top_k,
                            const float* top_p, const float* min_p, int joint,
                            const int64_t* seed, const int64_t* offset, const float* uniforms,
                            int32_t* tokens_out, double* probs_out, double* logprobs_out,
                            double* margin_out) {
  const int64_t rows = B * (int64_t)n_per_req;
  double* dist = (double*)malloc(sizeof(double) * (size_t)V);
  for (int64_t r = 0; r < rows; ++r) {
    const float* x = logits + r * ld;
    int64_t b = r / n_per_req;
    uint32_t j = (uint32_t)(r % n_per_req);
    float T = temperature ? temperature[r] : 1.0f;
    int32_t k = top_k ? top_k[r] : 0;
    float p = top_p ? top_p[r] : 1.0f;
    float mp = min_p ? min_p[r] : 0.0f;
    int64_t am = 0;
    double margin = orc_filter_row_ex(x, V, 1, T, k, p, mp, joint, dist, &am);
    float u = uniforms ? uniforms[r] : orc_verify_coin((uint64_t)seed[b], (uint64_t)offset[b], j);
    int64_t nnz = 0;
    double Z = 0.0;
    for (int64_t i = 0; i < V; ++i) {
      nnz += (dist[i] > 0.0);
      Z += dist[i];
    }
    double t = (double)u * Z;
    int64_t tok = -1, last_pos = -1;
    double S = 0.0;
    for (int64_t i = 0; i < V; ++i) {
      if (dist[i] > 0.0) {
        last_pos = i;
        if (S + dist[i] > t) {
          tok = i;
          if (nnz > 1) margin = dmin(margin, dmin(t - S, S + dist[i] - t) / Z);
          break;
        }
        S += dist[i];
      }
    }
    if (tok < 0) {
      tok = (last_pos >= 0) ? last_pos : am;
      margin = 0.0;
    }
    tokens_out[r] = (int32_t)tok;
    if (probs_out)
      for (int64_t i = 0; i < V; ++i) probs_out[r * V + i] = dist[i];
    if (logprobs_out) logprobs_out[r] = logprob_from_logits(x, V, tok);
    if (margin_out) margin_out[r] = margin;
  }
  free(dist);
}

/* Temperature-only draw by Gumbel-max (_sample_sharded_temperature: argmax of
 * l/T plus Gumbel noise is an exact sample of softmax(l/T); rows below the greedy
 * threshold stay greedy). Noise G = -ln(-ln u), u from the Gumbel Philox stream of
 * (request, row within request, token). Tokens with logit -inf never win.
 * margin_out[r] = (best - second best) / max(1, |best|). */
void orc_gumbel_max_sample(const float* logits, int64_t B, int32_t n_per_req,
                           int64_t V, int64_t ld, const float* temperature,
                           const int64_t* seed, const int64_t* offset,
                           int32_t* tokens_out, double* margin_out) {
  const int64_t rows = B * (int64_t)n_per_req;
  for (int64_t r = 0; r < rows; ++r) {
    const float* x = logits + r * ld;
    int64_t b = r / n_per_req;
    uint32_t n = (uint32_t)(r % n_per_req);
    float T = temperature ? temperature[r] : 1.0f;
    if (is_greedy(T)) {
      tokens_out[r] = (int32_t)orc_argmax(x, V);
      if (margin_out) margin_out[r] = INFINITY;
      continue;
    }
    double best = -INFINITY, second = -INFINITY;
    int64_t arg = -1;
    for (int64_t v = 0; v < V; ++v) {
      if (x[v] == -INFINITY) continue;
      float uu = orc_gumbel_u01((uint64_t)seed[b], (uint64_t)offset[b], n, (uint32_t)v);
      double g = -log(-log((double)uu));
      double s = (double)x[v] / (double)T + g;
      if (s > best) {
        second = best;
        best = s;
        arg = v;
      } else if (s > second) {
        second = s;
      }
    }
    if (arg < 0) arg = orc_argmax(x, V);
    tokens_out[r] = (int32_t)arg;
    if (margin_out) {
      double scale = fabs(best) > 1.0 ? fabs(best) : 1.0;
      margin_out[r] = (second == -INFINITY) ? INFINITY : (best - second) / scale;
    }
  }
}

/* out[r] = log_softmax(x[r])[t] at temperature 1 (logits) or ln x[r][t] (probs);
 * a token outside [0, V), -1 included, gives 0. */
void orc_gather_logprobs(const float* x, int is_probs, int64_t rows, int64_t V,
                         int64_t ld, const int32_t* tokens, double* out) {
  for (int64_t r = 0; r < rows; ++r) {
    int32_t t = tokens[r];
    if (t < 0 || (int64_t)t >= V) {
      out[r] = 0.0;
      continue;
    }
    const float* row = x + r * ld;
    out[r] = is_probs ? log((double)row[t]) : logprob_from_logits(row, V, t);
  }
}
