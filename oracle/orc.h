/*
 * Oracle for the speculative-decoding verify-and-sample step.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU
 * restatement of what the step computes, written so that each function can be
 * checked by eye against its definition. Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no
 * code, header or table with the CUDA library.
 *
 * Floating point: every probability, sum and logarithm is taken in double
 * (fp64) from the exact fp32 values of the inputs (bf16 inputs are widened to
 * fp32 by the caller, which is exact). The one exception is the accept test
 * with explicit fp32 probabilities, u*q < p, which the method states on fp32
 * values and which is therefore evaluated in fp32 here too.
 *
 * Sources, by page:
 *   [TS-FI]  TokenSpeed, sampling/backends/flashinfer.py: FlashInferSamplingBackend
 *            .sample() and .verify() (softmax with temperature, fused top-k/top-p
 *            renorm, verify_chain_greedy, chain_speculative_sampling_target_only,
 *            accept_length += 1, gather_token_logprobs_torch).
 *   [TRT-IF] TensorRT-LLM, _torch/speculative/interface.py: rejection_sampling_one_model
 *            docstring (tensor contract), SpecWorkerBase._sample_sharded_temperature
 *            (Gumbel-max is an exact temperature sample; rows below the greedy
 *            threshold stay greedy), greedy_argmax (lowest index on ties).
 *   Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
 *            (SC'11), for the Philox4x32-10 block function.
 *
 * Margins. Every floating-point decision also reports how far it was from
 * flipping, normalised to the quantity it compares (a probability or a total
 * mass). A GPU result that differs from the oracle's only where this margin
 * is below 1e-6 is a boundary case: counted and reported, not failed.
 */
#ifndef ORC_H
#define ORC_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Temperatures strictly below this are greedy (one-hot at the argmax). The
 * pages name a greedy temperature threshold without giving its value. */
#define ORC_GREEDY_T 1e-5f

/* Rows of a request at most (the library's limit on D is 64). */
#define ORC_MAX_R 65

/* ---- Philox4x32-10 and its streams --------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
float orc_u01(uint32_t x);
float orc_verify_coin(uint64_t seed, uint64_t offset, uint32_t j);
float orc_gumbel_u01(uint64_t seed, uint64_t offset, uint32_t n, uint32_t v);

/* ---- Row-level definitions ----------------------------------------------- */
int64_t orc_argmax(const float* x, int64_t V);
double orc_filter_row(const float* vals, int64_t V, int is_logits, float T,
                      int32_t top_k, float top_p, double* out, int64_t* argmax_out);
double orc_filter_row_ex(const float* vals, int64_t V, int is_logits, float T,
                         int32_t top_k, float top_p, float min_p, int joint, double* out,
                         int64_t* argmax_out);

/* ---- The six operations -------------------------------------------------- */
void orc_softmax_temp(const float* logits, int64_t rows, int64_t V, int64_t ld,
                      const float* temperature, double* probs_out);
void orc_topk_topp_renorm(const float* probs, int64_t rows, int64_t V, int64_t ld,
                          const int32_t* top_k, const float* top_p, double* out,
                          double* margin_out);
void orc_verify_chain_greedy(const float* logits, int64_t B, int32_t D, int64_t V,
                             int64_t ld, const int32_t* draft_tokens,
                             int32_t* accepted_tokens, int32_t* accept_length,
                             int32_t* accept_index, double* logprobs);
void orc_chain_spec_sampling(const float* target, int target_is_logits, int64_t B,
                             int32_t D, int64_t V, int64_t ld,
                             const float* temperature, const int32_t* top_k,
                             const float* top_p, const float* draft_probs,
                             int64_t ld_draft, const int32_t* draft_tokens,
                             const int64_t* seed, const int64_t* offset,
                             const float* uniforms, int32_t* accepted_tokens,
                             int32_t* accept_length, int32_t* accept_index,
                             double* logprobs, double* margin_out);
void orc_gumbel_max_sample(const float* logits, int64_t B, int32_t n_per_req,
                           int64_t V, int64_t ld, const float* temperature,
                           const int64_t* seed, const int64_t* offset,
                           int32_t* tokens_out, double* margin_out);
void orc_gather_logprobs(const float* x, int is_probs, int64_t rows, int64_t V,
                         int64_t ld, const int32_t* tokens, double* out);

/* ---- The next rows: single-step sampling, min_p, relaxed acceptance ------ */
void orc_chain_spec_sampling_ex(const float* target, int target_is_logits, int64_t B,
                                int32_t D, int64_t V, int64_t ld, const float* temperature,
                                const int32_t* top_k, const float* top_p, const float* min_p,
                                float threshold_single, float threshold_acc,
                                const float* draft_probs, int64_t ld_draft,
                                const int32_t* draft_tokens, const int64_t* seed,
                                const int64_t* offset, const float* uniforms,
                                int32_t* accepted_tokens, int32_t* accept_length,
                                int32_t* accept_index, double* logprobs, double* margin_out);
void orc_verify_chain_greedy_ragged(const float* logits, int64_t B, int32_t D, int64_t V,
                                    int64_t ld, const int32_t* qo_indptr,
                                    const int32_t* draft_tokens, int32_t* accepted_tokens,
                                    int32_t* accept_length, int32_t* accept_index,
                                    double* logprobs);
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
                                    double* margin_out);
void orc_sample_from_logits(const float* logits, int64_t B, int32_t n_per_req, int64_t V,
                            int64_t ld, const float* temperature, const int32_t* top_k,
                            const float* top_p, const float* min_p, int joint,
                            const int64_t* seed, const int64_t* offset, const float* uniforms,
                            int32_t* tokens_out, double* probs_out, double* logprobs_out,
                            double* margin_out);

#ifdef __cplusplus
}
#endif
#endif
