/*
 * ts_verify.h - C ABI of libtsverify.so: the speculative-decoding verify-and-sample
 * step on one GB300 (sm_103a) GPU.
 *
 * What the step computes is defined by three public pages:
 *   [TS-FI]  TokenSpeed, runtime/sampling/backends/flashinfer.py,
 *            FlashInferSamplingBackend.verify() / .sample();
 *   [TS-DP]  TokenSpeed, runtime/distributed/dp_sampling_comm.py (output layout);
 *   [TRT-IF] TensorRT-LLM, _torch/speculative/interface.py,
 *            rejection_sampling_one_model(), SpecWorkerBase._sample_sharded_temperature().
 *
 * Conventions for every call
 * --------------------------
 *  - Pointers named *_host are host memory; every other pointer is CUDA device memory
 *    owned by the caller. The library never allocates, frees or synchronises: each
 *    call enqueues its kernels on `stream` and returns.
 *  - Rows: a [batch, R, vocab] tensor is rows b*R + j of a row-major matrix whose rows
 *    are `ld` elements apart (ld >= vocab). R = D + 1 for verification.
 *  - Token ids are int32; seeds and offsets int64; probabilities fp32. Logits are fp32
 *    or bf16 (TS_F32 / TS_BF16); bf16 is widened to fp32 exactly.
 *  - Knobs: temperature < TS_GREEDY_T (or NaN) means greedy (one-hot at the argmax);
 *    top_k <= 0 or >= vocab means no top-k; top_p >= 1 means no top-p. A NULL knob
 *    array means "off" (temperature 1).
 *  - Ties: the argmax and top-k keep the lowest token id among equal values.
 *  - Workspace: calls that need scratch take `workspace`/`ws_bytes`, a caller-owned
 *    device buffer of at least ts_workspace_size(...) bytes that must be zero-filled
 *    once before its first use (ts_workspace_init does that). Every call leaves the
 *    counters it keeps there at zero again (the rest is scratch), so it can be reused
 *    by later calls on the same stream without clearing. Calls that overlap on the GPU
 *    must not share a workspace.
 *  - Errors: arguments are validated on the host before any launch; an invalid call
 *    returns TS_ERR_INVALID_ARG / TS_ERR_UNSUPPORTED_DTYPE and enqueues nothing. A
 *    failed launch returns TS_ERR_CUDA. ts_last_error_message() (thread-local) gives
 *    the reason for the last failure of the calling thread.
 *  - Limits: 1 <= vocab <= TS_MAX_VOCAB, 0 <= D <= TS_MAX_DRAFT, batch >= 1. Rows the
 *    streaming kernels cannot take (not 16-byte aligned, or longer than they stage)
 *    go to a cluster-staged kernel that holds at most 655360 bf16 / 327680 fp32
 *    tokens a row: ts_softmax_temp, ts_topk_topp_renorm and ts_chain_spec_sampling
 *    reject larger such rows with TS_ERR_INVALID_ARG.
 *  - Inputs with NaN are outside the contract (no fault; results unspecified).
 */
#ifndef TS_VERIFY_H
#define TS_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,
  TS_ERR_UNSUPPORTED_DTYPE = 2,
  TS_ERR_CUDA = 3,
  TS_ERR_TIMEOUT = 4 /* a bounded device-side wait gave up (see ts_device_error) */
} ts_status;

typedef enum { TS_F32 = 0, TS_BF16 = 1 } ts_dtype;

#define TS_GREEDY_T 1e-5f
#define TS_MAX_DRAFT 64
#define TS_MAX_VOCAB (1 << 22)

/* Bytes of workspace any call below needs for `batch` requests of `rows_per_req` rows
 * over `vocab` tokens (rows_per_req = D + 1 for verification, n_per_req for
 * ts_gumbel_max_sample, 1 for per-row calls with batch = rows). */
size_t ts_workspace_size(int64_t batch, int32_t rows_per_req, int64_t vocab);

/* Zero-fills a workspace on `stream` (cudaMemsetAsync). */
ts_status ts_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream);

/* The reason for the calling thread's last non-OK status ("" if none). */
const char* ts_last_error_message(void);

/* Synchronises the current device and reads (then, if clear != 0, clears) the
 * library's device error word: 0 if no bounded wait ever gave up; otherwise bits 0-7
 * come from the cluster-staged kernels, bits 8-15 from the renorm row kernel, bits
 * 16-23 from the staged softmax and bits 24-31 from the chain kernel (bit 24: a stage
 * wait gave up; bit 25: a CTA's wait for its own copies in flight ran out). The word is
 * sticky until cleared, but it only reports: a later call is not affected by it.
 * Returns TS_ERR_TIMEOUT if a wait gave up, TS_ERR_CUDA if the read failed. A
 * diagnostic, not part of the hot path. */
ts_status ts_device_error(uint32_t* word_host, int clear);

/* Sets how many SM clock cycles a stage wait of the chain kernel (ts_chain_spec_sampling
 * from logits) may take before it gives up; 0 restores the default of 2^32 (about 2 s).
 * Process-wide; takes effect for calls enqueued afterwards. A CTA whose wait gives up
 * issues no more copies, waits (on the long budget) for the copies it has in flight,
 * and leaves the requests it had not finished with accept_length = 0; their other
 * outputs are unspecified. ts_device_error then reports TS_ERR_TIMEOUT. A diagnostic:
 * it exists so that this path can be tested. */
ts_status ts_set_wait_cycles(uint64_t cycles);

/* Temperature softmax [TS-FI verify(): softmax(logits, temperature)].
 * probs_out[r, i] = exp((x_ri - M_r)/T_r) / sum_k exp((x_rk - M_r)/T_r), M_r the row max;
 * one-hot at the row argmax when T_r < TS_GREEDY_T. temperature: [rows] or NULL (= 1).
 * logits: [rows, ld] of `dt`; probs_out: [rows, vocab] fp32, contiguous, must not alias
 * logits. */
ts_status ts_softmax_temp(const void* logits, ts_dtype dt, int64_t rows, int64_t vocab,
                          int64_t ld, const float* temperature, float* probs_out,
                          cudaStream_t stream);

/* Top-k then top-p renormalisation of probability rows, fused [TS-FI verify():
 * fused_topk_topp_renorm, the replacement for top_k_renorm_prob followed by
 * top_p_renorm_prob]. Top-k keeps the k largest probabilities (exactly k; lowest ids
 * first among equals); top-p then keeps, in the same order, each token whose
 * preceding kept mass is below top_p times the kept mass (the first token always).
 * The result is renormalised; dropped tokens are 0.
 * probs: [rows, ld] fp32 (non-negative); top_k: [rows] or NULL; top_p: [rows] or NULL;
 * probs_out: [rows, vocab] fp32 contiguous; may equal probs when ld == vocab. A row
 * whose kept tokens carry no mass (in 2^-40 units of the row) is written as zeros. */
ts_status ts_topk_topp_renorm(const float* probs, int64_t rows, int64_t vocab, int64_t ld,
                              const int32_t* top_k, const float* top_p, float* probs_out,
                              cudaStream_t stream);

/* Greedy chain verification [TS-FI verify(): sampling_argmax then verify_chain_greedy;
 * TRT-IF strict acceptance]. Draft j of request b is accepted while it equals the
 * argmax of target row (b, j); the argmax of the first mismatching row (or of row D,
 * the bonus) follows.
 * target_logits: [batch*(D+1), ld] of `dt`; draft_tokens: [batch, D].
 * Out: accepted_tokens [batch, D+1] (accepted drafts, the target token, then -1),
 * accept_length [batch] in [1, D+1] (tokens emitted), accept_index [batch, D+1]
 * (b*(D+1)+j for emitted positions, else -1; NULL = skip), logprobs [batch, D+1]
 * (log-softmax at temperature 1 of the raw logits at each emitted token, 0 after;
 * NULL = skip). */
ts_status ts_verify_chain_greedy(const void* target_logits, ts_dtype dt, int64_t batch,
                                 int32_t D, int64_t vocab, int64_t ld,
                                 const int32_t* draft_tokens, int32_t* accepted_tokens,
                                 int32_t* accept_length, int32_t* accept_index,
                                 float* logprobs, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream);

/* Greedy verification of a ragged batch [TRT-IF ragged_helpers count_accepted_ragged,
 * scatter_ragged_to_padded: each request verifies its own window]: as
 * ts_verify_chain_greedy, with the target rows packed as described for
 * ts_chain_args.qo_indptr (request b owns rows qo_indptr[b] .. qo_indptr[b+1] - 1, at
 * most D + 1 of them, and compares its first L_b - 1 drafts), total_rows rows in all,
 * drafts [batch, D] padded, outputs [batch, D+1] padded, accept_index packed row numbers.
 * The outputs are cleared on `stream` first (accept_length 0, tokens and indices -1,
 * logprobs 0), which is what a window that does not fit leaves.
 * Workspace: ts_workspace_size(batch, D + 1, vocab). */
ts_status ts_verify_chain_greedy_ragged(const void* target_logits, ts_dtype dt, int64_t batch,
                                        int32_t D, int64_t vocab, int64_t ld,
                                        const int32_t* qo_indptr, int64_t total_rows,
                                        const int32_t* draft_tokens, int32_t* accepted_tokens,
                                        int32_t* accept_length, int32_t* accept_index,
                                        float* logprobs, void* workspace, size_t ws_bytes,
                                        cudaStream_t stream);

/* Arguments of ts_chain_spec_sampling. Layouts as in the comments; NULL where allowed. */
typedef struct ts_chain_args {
  const void* target;        /* [batch*(D+1), ld]: logits (target_is_logits = 1, dtype
                                target_dtype) or fp32 probabilities (target_is_logits = 0) */
  int32_t target_dtype;      /* ts_dtype; must be TS_F32 for probabilities */
  int32_t target_is_logits;
  int64_t batch;
  int32_t D;
  int32_t reserved0;
  int64_t vocab;
  int64_t ld;
  const float* temperature;  /* [batch] or NULL; logits only */
  const int32_t* top_k;      /* [batch] or NULL; logits only */
  const float* top_p;        /* [batch] or NULL; logits only */
  const float* draft_probs;  /* [batch*D, ld_draft] fp32, or NULL: target-only (the draft
                                is a point mass on the drafted token). With logit targets
                                the rows must be 16-byte aligned and vocab <= 2^18 (else
                                TS_ERR_INVALID_ARG) */
  int64_t ld_draft;
  const int32_t* draft_tokens; /* [batch, D]; ids outside [0, vocab) are never accepted */
  const int64_t* seed;       /* [batch] Philox key (two's-complement bits) */
  const int64_t* offset;     /* [batch] Philox counter base */
  const float* uniforms;     /* [batch, D+1] explicit coins in (0, 1) replacing Philox:
                                u_j for the test at j < D, u_D for the final draw; or NULL */
  int32_t* accepted_tokens;  /* [batch, D+1] out */
  int32_t* accept_length;    /* [batch] out */
  int32_t* accept_index;     /* [batch, D+1] out, or NULL */
  float* logprobs;           /* [batch, D+1] out, or NULL: logits: log-softmax at T = 1 of
                                the raw row; probabilities: ln p(token); 0 after the last
                                emitted token */
  /* Added knobs; a zero-initialised struct keeps the plain method. Both need logit
   * targets with 16-byte aligned rows and vocab <= 2^18 (else TS_ERR_INVALID_ARG). */
  const float* min_p;        /* [batch] or NULL: of the tokens top-k and top-p keep, only
                                those with p_i >= min_p * max_i p_i stay (min_p clamped to
                                [0, 1]; TRT-IF fused_sample_from_logits min_ps) */
  float threshold_single;    /* relaxed acceptance (TS-FI verify() threshold_single and */
  float threshold_acc;       /* threshold_acc), target-only: accept iff p(x) >= t_single
                                or u * t_acc < p(x). Values outside (0, 1) mean 1 (plain
                                rejection sampling); not allowed with draft_probs. */
  /* Ragged verification (TRT-IF SpecMetadata verify_lens / qo_indptr), or NULL: the
   * target rows are packed, request b owning rows qo_indptr[b] .. qo_indptr[b+1] - 1
   * (L_b of them, 1 <= L_b <= D + 1) and verifying its first L_b - 1 drafts exactly as a
   * request with D = L_b - 1 would; total_rows = qo_indptr[batch] rows in all. Drafts,
   * draft probabilities and coins keep the padded [batch, D(+1)] layouts (the final
   * draw's coin is position L_b - 1 of the request's stream, or uniforms[b, L_b - 1]);
   * outputs are [batch, D+1] with -1 (tokens, indices) and 0 (logprobs) past the
   * emitted tokens, and accept_index holds packed row numbers qo_indptr[b] + j. A window
   * outside [1, D + 1] rows or past total_rows leaves its request at accept_length 0.
   * Logit targets only, 16-byte aligned rows, vocab <= 2^18 (else TS_ERR_INVALID_ARG). */
  const int32_t* qo_indptr;  /* [batch + 1] device, or NULL */
  int64_t total_rows;
} ts_chain_args;

/* Chain speculative sampling [TRT-IF rejection_sampling_one_model; TS-FI verify():
 * softmax + fused top-k/top-p renorm + chain_speculative_sampling_target_only].
 * p_j is the target distribution of row (b, j): softmax(logits/T) renormalised by top-k
 * and top-p (logits), or the given row (probabilities). For j = 0..D-1 with draft x_j:
 *   with draft probs q: accept iff u_j * q_j(x_j) < p_j(x_j)  (accept w.p. min(1, p/q));
 *   target-only:        accept iff u_j < p_j(x_j).
 * At the first rejection j*, the token is drawn from norm(max(p_j* - q_j*, 0))
 * (target-only: p_j* with x_j* removed); if all D drafts are accepted, the bonus is
 * drawn from p_D. The draw uses u_D: the smallest token id whose inclusive prefix mass,
 * in token-id order, exceeds u_D times the total mass. With explicit probabilities the
 * accept test is evaluated in fp32 (one rounded product); the residual max(p - q, 0) is
 * formed elementwise in fp32. With logits and draft probabilities, p is the filtered
 * distribution of the logits (temperature, top-k, top-p), the accept test compares
 * u q(x) with p(x) in double, and the residual max(p - q, 0) of the rejected row is formed
 * elementwise in fp32 from p's fixed-point weights.
 * Coins: uniforms if given, else Philox4x32-10 keyed by seed[b] with counter
 * (j, 0xFFFFFFFF, lo32(offset[b]), hi32(offset[b])), word 0 mapped to
 * (2*(w >> 9) + 1) * 2^-24.
 * Outputs as ts_verify_chain_greedy. */
ts_status ts_chain_spec_sampling(const ts_chain_args* args, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream);

/* Arguments of ts_sample_from_logits. rows = batch * n_per_req; row r belongs to request
 * r / n_per_req as its row j = r % n_per_req. */
#define TS_FILTER_TOP_K_FIRST 0 /* top-p measured on the top-k renormalised distribution */
#define TS_FILTER_JOINT 1       /* top-k and top-p both measured on the unfiltered one */
typedef struct ts_sample_args {
  const void* logits;        /* [rows, ld], dtype */
  int32_t dtype;             /* ts_dtype */
  int32_t n_per_req;         /* rows of a request (>= 1) */
  int64_t batch;
  int64_t vocab;
  int64_t ld;
  const float* temperature;  /* [rows] or NULL (1); below TS_GREEDY_T: the argmax */
  const int32_t* top_k;      /* [rows] or NULL */
  const float* top_p;        /* [rows] or NULL */
  const float* min_p;        /* [rows] or NULL (see ts_chain_args.min_p) */
  int32_t filter_order;      /* TS_FILTER_TOP_K_FIRST or TS_FILTER_JOINT */
  int32_t reserved0;
  const int64_t* seed;       /* [batch] Philox key */
  const int64_t* offset;     /* [batch] Philox counter base */
  const float* uniforms;     /* [rows] explicit coins in (0, 1) replacing Philox, or NULL */
  int32_t* tokens;           /* [rows] out */
  float* logprobs;           /* [rows] out, or NULL: log-softmax at T = 1 of the raw row */
  float* probs;              /* out, or NULL: row r's kept distribution (0 outside it, fp32)
                                at probs + dst * ld_probs, dst = probs_row ? probs_row[r] : r */
  int64_t ld_probs;          /* >= vocab */
  const int64_t* probs_row;  /* [rows] destination rows, or NULL */
} ts_sample_args;

/* Single-step sampling from logits [TS-FI sample(): softmax(logits, temperature), then
 * top_k_top_p_sampling_from_probs(..., filter_apply_order="joint", seed, offset);
 * TRT-IF advanced_sample_draft / advanced_sample_draft_block:
 * fused_sample_from_logits_with_probs(logits, temperatures, top_ks, top_ps, min_ps, seed,
 * offset), the probabilities stored for the next verify step]. Each row's distribution
 * is filtered as ts_chain_spec_sampling's p (in filter_order; min_p last) and one token
 * is drawn by the inverse CDF in token-id order with coin u: uniforms[r], else the coin
 * of position j of request b's stream as in ts_chain_spec_sampling (Philox keyed by
 * seed[b], counter (j, 0xFFFFFFFF, lo32(offset[b]), hi32(offset[b]))). Draft-side calls
 * and the verify call that checks their drafts must therefore use different offsets.
 * Rows must be 16-byte aligned and vocab <= 2^18 (else TS_ERR_INVALID_ARG). Workspace:
 * ts_workspace_size(batch * n_per_req, 1, vocab). */
ts_status ts_sample_from_logits(const ts_sample_args* args, void* workspace, size_t ws_bytes,
                                cudaStream_t stream);

/* Temperature-only sampling by Gumbel-max [TRT-IF _sample_sharded_temperature: the
 * argmax of x/T plus Gumbel noise is an exact sample of softmax(x/T); rows below the
 * greedy threshold stay greedy]. rows = batch * n_per_req; row r belongs to request
 * r / n_per_req as its row n = r % n_per_req. tokens_out[r] = argmax_i (x_ri/T_r + G_ri),
 * G = -ln(-ln u), u from Philox4x32-10 keyed by seed[b], counter (i >> 2, n,
 * lo32(offset[b]), hi32(offset[b])), word i & 3, mapped as for the coins. Tokens with
 * logit -inf never win. temperature: [rows]; seed, offset: [batch]. */
ts_status ts_gumbel_max_sample(const void* logits, ts_dtype dt, int64_t batch,
                               int32_t n_per_req, int64_t vocab, int64_t ld,
                               const float* temperature, const int64_t* seed,
                               const int64_t* offset, int32_t* tokens_out, void* workspace,
                               size_t ws_bytes, cudaStream_t stream);

/* Chosen-token logprobs [TS-FI gather_token_logprobs_torch]:
 * out[r] = log_softmax(x[r, :])[tokens[r]] at temperature 1 (is_probs = 0) or
 * ln x[r, tokens[r]] (is_probs = 1, fp32 only); a token outside [0, vocab) gives 0.
 * x: [rows, ld]; tokens: [rows]; out: [rows] fp32. */
ts_status ts_gather_logprobs(const void* x, ts_dtype dt, int32_t is_probs, int64_t rows,
                             int64_t vocab, int64_t ld, const int32_t* tokens, float* out,
                             void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Greedy chain verification that allocates nothing and takes no workspace. The pages
 * have no counterpart: this entry point exists for callers that cannot give the library
 * device memory, such as a host binding the C ABI without a device allocator of its own,
 * or code whose device memory is a fixed budget owned by another allocator. Same
 * arguments, outputs and semantics as ts_verify_chain_greedy, minus workspace/ws_bytes.
 * Scratch: a file-scope device array of 4 MiB; every GPU that loads the library holds
 * its own copy until the process exits. Calls with batch*(D+1) > TS_STATIC_MAX_ROWS are
 * rejected with TS_ERR_INVALID_ARG. Each call looks up the array's device address on the
 * current device (cudaGetSymbolAddress, which allocates nothing); the first call on a
 * device also loads the library's device code there, so make that first call before any
 * stream capture. Each call clears the array's arrival counters on `stream`
 * (cudaMemsetAsync) and calls no allocating routine. All calls on one device share that
 * device's copy of the array: calls that may overlap on the same device (different
 * streams or host threads) race and must be serialised by the caller. */
#define TS_STATIC_MAX_ROWS 2048
ts_status ts_verify_chain_greedy_static(const void* target_logits, ts_dtype dt, int64_t batch,
                                        int32_t D, int64_t vocab, int64_t ld,
                                        const int32_t* draft_tokens, int32_t* accepted_tokens,
                                        int32_t* accept_length, int32_t* accept_index,
                                        float* logprobs, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TS_VERIFY_H */
