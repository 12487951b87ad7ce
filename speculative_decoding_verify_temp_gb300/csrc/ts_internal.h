// Internal interface between the C ABI (ts_abi.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tsv {

constexpr int kMaxSplits = 64;  // row splits of the streaming kernels
constexpr int kSTopK = 1024;  // largest top_k the row kernel's candidate lists serve
constexpr int kSVecs = 8;     // 16-byte vectors a thread covers in a 32 KB chunk
constexpr int kSThreads = 256;

// 32 KB chunks (256 threads x 8 vectors) of a row of V elements of `esize` bytes: the row
// kernel keeps kSTopK workspace slots per chunk for a row (per-range masses of its
// plain and top-p rows). Returns false if a row needs more than kMaxSplits chunks.
inline bool sample_splits(int64_t V, int esize, int32_t* splits, int64_t* chunk) {
  const int64_t c = (int64_t)kSThreads * kSVecs * (16 / esize);
  *chunk = c;
  const int64_t s = (V + c - 1) / c;
  *splits = (int32_t)(s < kMaxSplits ? s : kMaxSplits);
  return s <= kMaxSplits;
}

// Per-(row, split) partial of the streaming row statistics: argmax (v, i) and the
// log-sum-exp state s * exp(m) of the raw row.
struct alignas(16) Part {
  float v;
  int32_t i;
  float m;
  float s;
};

// Per-row result handed from the row kernels to the request-level chain writer.
struct alignas(64) RowRes {
  float M;       // row maximum (raw logits)
  int32_t am;    // row argmax
  float S;       // sum exp(x - M) at temperature 1 (logprobs), or 0
  int32_t tok;   // drawn token of this row (residual or bonus draw), -1 if none
  int32_t acc;   // 1 if the draft of this row was accepted
  int32_t pad[3];
  // the chain kernel's kept set, for a residual draw against draft probabilities:
  uint64_t C;    // threshold composite (a token is kept iff its composite >= C)
  uint64_t Zk;   // kept mass in 2^-40 units of the maximum's weight
  int32_t gh, gl;  // top-p rows: sixteenths above gh are kept, gl..gh by C
  int32_t kind;    // 0 greedy (the argmax), 1 by C, 2 every token, 3 top-p window + C
  int32_t pad2;
};

// Per-request partial of the streaming draw: residual mass and base mass.
struct alignas(8) DrawPart {
  float w;
  float b;
};

// Workspace carve-up for `batch` requests of `R` rows each.
struct Workspace {
  uint32_t* rowcnt;   // [rows]
  uint32_t* reqcnt;   // [batch]
  Part* part;         // [rows * kMaxSplits]
  RowRes* rowres;     // [rows]
  DrawPart* dpart;    // [batch * kMaxSplits]
  uint64_t* cmass;    // [rows * 8] per-CTA masses of a cluster-staged row
  uint32_t* best;     // [rows] Gumbel-max: the row's best score so far (order key, 0: none)
  uint32_t* work;     // [4] the row kernel's 64-bit next-row counter ([0..1], 8-byte
                      // aligned) and finished-CTA count ([2]); the chain kernel's count
                      // of rows served by its general path ([2]) and row claims ([3])
  uint32_t* order;    // [rows] the chain kernel's rows in claim order (cost tiers)
  uint32_t* creq;     // [batch] the chain kernel's per-request finished-row counts
  int32_t* slen;      // [batch] single-step sampling: the chain kernel's accept lengths
  uint32_t* rreq;     // [rows] ragged verification: the request of each packed row
  uint64_t* cand;     // [rows * cand_splits * kSTopK] per-row range masses of the row
                      // kernel (vocab > 0 only)
  int64_t cand_splits;
  size_t bytes;
};

// vocab = 0 lays out no candidate lists.
size_t workspace_layout(int64_t batch, int32_t R, int64_t vocab, void* base, Workspace* ws);

// ---- streaming kernels (ts_stream.cu) ------------------------------------------

struct RowStatArgs {
  const void* x;
  int64_t ld, V, rows;
  int32_t splits;
  int64_t split_len;  // elements per split, a multiple of 8
  int32_t vec;        // rows are 16-byte aligned
  int32_t want_lse;
  int32_t kind;       // 0: greedy verify, 1: gather logprobs (logits), 2: Gumbel-max
  // Gumbel
  const float* temperature;
  const int64_t* seed;
  const int64_t* offset;
  int32_t n_per_req;
  int32_t* tokens_out;
  // greedy verify
  int32_t D;
  const int32_t* draft_tokens;
  int32_t* accepted_tokens;
  int32_t* accept_length;
  int32_t* accept_index;
  float* logprobs;
  // greedy verify inside a sampled chain: rows of requests whose temperature (per
  // request) is not greedy are left to the staged kernel
  const float* req_temperature;
  // gather logprobs
  const int32_t* lp_tokens;
  float* lp_out;
  Workspace ws;
  // greedy verify of a ragged batch: request b owns the packed rows qo[b] .. qo[b+1] - 1
  // (at most D + 1; rows = their total); NULL: rows b (D+1) ..
  const int32_t* qo;
  int64_t nreq;
};

cudaError_t launch_rowstat(const RowStatArgs& a, int bf16, cudaStream_t s);

// ---- Gumbel-max over 16-byte aligned rows (ts_gumbel.cu) -----------------------------

struct GumbelArgs {
  const void* x;
  int64_t ld, V, rows;
  int32_t n_per_req;
  const float* temperature;  // [rows]
  const int64_t* seed;       // [rows / n_per_req]
  const int64_t* offset;     // [rows / n_per_req]
  int32_t* tokens_out;       // [rows]
  int64_t chunk_vecs;        // 16-byte vectors a chunk (the last chunk of a row may be shorter)
  int32_t cpr;               // chunks a row (<= kMaxSplits); the last also takes the ragged tail
  uint32_t total_chunks;     // rows * cpr
  int32_t grid;              // persistent CTAs
  Workspace ws;              // rowcnt, part, best (left zero) and work[0] (claims)
};

cudaError_t launch_gumbel(const GumbelArgs& a, int bf16, cudaStream_t s);
int gumbel_ctas_per_sm(int bf16);

struct DrawArgs {
  const float* p;
  int64_t ld, V, B;
  int32_t D;
  const float* q;
  int64_t ld_q;
  const int32_t* drafts;
  const int64_t* seed;
  const int64_t* offset;
  const float* uniforms;
  int32_t splits;
  int64_t split_len;
  int32_t vec;
  int32_t* accepted_tokens;
  int32_t* accept_length;
  int32_t* accept_index;
  float* logprobs;
  Workspace ws;
};

cudaError_t launch_draw_probs(const DrawArgs& a, cudaStream_t s);

// Temperature softmax of 16-byte aligned rows into [rows, V] fp32 (ts_stream.cu).
cudaError_t launch_softmax(const void* x, int bf16, int64_t rows, int64_t ld, int64_t V,
                           const float* temperature, float* out, cudaStream_t s);
cudaError_t softmax_read_error(uint32_t* word, int clear);

cudaError_t launch_logprobs_probs(const float* p, int64_t ld, int64_t V, int64_t rows,
                                  const int32_t* tokens, float* out, cudaStream_t s);

// ---- row-streaming kernel (ts_sample.cu) -----------------------------------------

// Arguments of the row-streaming kernels: the renorm of probability rows (ts_sample.cu)
// and target-only chain sampling from logits (ts_chain.cu). Both require 16-byte aligned
// rows and vocab <= kRowMaxVocab.
struct SampleArgs {
  const void* x;
  int32_t bf16;
  int64_t ld, V, rows;
  int32_t R, D;
  int32_t splits;
  int64_t chunk;  // elements per chunk
  const float* temperature;  // per request
  const int32_t* top_k;
  const float* top_p;
  const int32_t* draft_tokens;
  const int64_t* seed;
  const int64_t* offset;
  const float* uniforms;
  int32_t* accepted_tokens;
  int32_t* accept_length;
  int32_t* accept_index;
  float* logprobs;
  Workspace ws;
  float* out;  // top-k/top-p renorm of probability rows: [rows, V] fp32 (no workspace)
  uint64_t wait_cycles;  // chain kernel: SM clock cycles a stage wait may take
  const float* q;        // chain kernel: draft probabilities [B*D, ld_q] fp32, or NULL
  int64_t ld_q;
  // chain kernel, the next rows
  const float* min_p;    // per request (per row when sampling), or NULL
  int32_t joint;         // top-p measured on the whole row's mass (single-step sampling)
  float thr_single;      // relaxed acceptance (1: plain rejection sampling)
  float thr_acc;
  int32_t sample_n;      // 0: chain verification; > 0: single-step sampling of rows in
                         // requests of sample_n rows (R = 1, D = 0; knobs per row, seed and
                         // offset per request, coin row % sample_n)
  float* probs_out;      // sampling: the kept distribution of each row, or NULL
  int64_t ld_probs;
  const int64_t* probs_row;  // destination row of each row's distribution, or NULL
  // ragged verification: request b owns the packed rows qo[b] .. qo[b + 1] - 1 (at most
  // R of them); NULL: request b owns rows b R .. b R + R - 1. Outputs stay [nreq, R].
  const int32_t* qo;
  int64_t nreq;
};

// The row kernel in its renorm mode (fp32 probability rows, 16-byte aligned).
cudaError_t launch_renorm_rows(const SampleArgs& a, cudaStream_t s);
cudaError_t row_read_error(uint32_t* word, int clear);

// ---- chain kernel (ts_chain.cu) -----------------------------------------------------

// Target-only chain sampling from logits (16-byte aligned rows, vocab <= kRowMaxVocab):
// a planning launch orders the rows by cost tier and clears the per-launch state, then a
// persistent row-streaming launch serves every row.
cudaError_t launch_chain(const SampleArgs& a, cudaStream_t s);
cudaError_t chain_read_error(uint32_t* word, int clear);
constexpr int64_t kRowMaxVocab = (int64_t)1 << 18;  // the row kernel's exact digit sums

// ---- cluster-staged row kernels (ts_staged.cu) -----------------------------------

enum StagedMode { kSoftmax = 0, kRenorm = 1, kChain = 2 };

struct StagedArgs {
  int32_t mode;
  const void* x;
  int32_t bf16;
  int64_t ld, V, rows;
  int32_t R, D;  // chain: rows per request and drafts
  const float* temperature;  // softmax: per row; chain: per request
  const int32_t* top_k;      // renorm: per row; chain: per request
  const float* top_p;
  float* out;  // softmax / renorm output, [rows, V]
  // chain (target-only, logits)
  const int32_t* draft_tokens;
  const int64_t* seed;
  const int64_t* offset;
  const float* uniforms;
  int32_t* accepted_tokens;
  int32_t* accept_length;
  int32_t* accept_index;
  float* logprobs;
  int32_t skip_greedy;  // chain: greedy requests are handled by the streaming kernel
  Workspace ws;
};

cudaError_t launch_staged(const StagedArgs& a, cudaStream_t s, const char** why);
cudaError_t staged_read_error(uint32_t* word, int clear);
int staged_max_vocab(int bf16);

}  // namespace tsv
