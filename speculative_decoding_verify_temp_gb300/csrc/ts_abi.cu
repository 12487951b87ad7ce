// The C ABI of libtsverify.so: argument validation, workspace carve-up, launch geometry
// and dispatch to the kernels. Host code only; every step of the computation runs in
// the kernels of ts_stream.cu, ts_sample.cu and ts_staged.cu.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>

#include <cuda_runtime.h>

#include "../../include/ts_verify.h"
#include "ts_internal.h"

namespace {

thread_local char g_msg[512] = "";

// SM clock cycles a stage wait of the chain kernel may take before it gives up.
constexpr uint64_t kDefaultWaitCycles = (uint64_t)1 << 32;
std::atomic<uint64_t> g_wait_cycles{kDefaultWaitCycles};

ts_status fail(ts_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

ts_status cuda_fail(cudaError_t e, const char* what) {
  return fail(TS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void* p, int64_t ld, int esize) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esize) % 16 == 0);
}

// Splits of a row so that about 8 CTAs per SM are in flight, each streaming >= min_len.
void choose_splits(int64_t units, int64_t V, int64_t min_len, int32_t* splits, int64_t* len) {
  const int64_t target = (int64_t)sm_count() * 8;
  int64_t s = (target + units - 1) / units;
  s = s < 1 ? 1 : (s > tsv::kMaxSplits ? tsv::kMaxSplits : s);
  const int64_t smax = (V + min_len - 1) / min_len;
  if (s > smax) s = smax < 1 ? 1 : smax;
  int64_t l = ((V + s - 1) / s + 7) & ~(int64_t)7;
  *len = l;
  *splits = (int32_t)((V + l - 1) / l);
}

// A threshold in (0, 1) relaxes the accept test; any other value (0 from a
// zero-initialised struct, 1, NaN) means 1.
float unit_threshold(float t) { return (t > 0.f && t < 1.f) ? t : 1.f; }

ts_status check_common(int64_t rows, int64_t V, int64_t ld) {
  if (rows < 1) return fail(TS_ERR_INVALID_ARG, "rows/batch must be >= 1 (got %lld)", (long long)rows);
  if (V < 1 || V > TS_MAX_VOCAB)
    return fail(TS_ERR_INVALID_ARG, "vocab must be in [1, %d] (got %lld)", TS_MAX_VOCAB, (long long)V);
  if (ld < V) return fail(TS_ERR_INVALID_ARG, "ld (%lld) must be >= vocab (%lld)", (long long)ld, (long long)V);
  if (rows > (int64_t)1 << 30) return fail(TS_ERR_INVALID_ARG, "too many rows");
  return TS_OK;
}

ts_status check_dtype(int dt) {
  if (dt != TS_F32 && dt != TS_BF16) return fail(TS_ERR_UNSUPPORTED_DTYPE, "unsupported dtype %d", dt);
  return TS_OK;
}

ts_status take_workspace(int64_t batch, int32_t R, int64_t vocab, void* ws, size_t ws_bytes,
                         tsv::Workspace* out) {
  const size_t need = tsv::workspace_layout(batch, R, vocab, ws, out);
  if (ws == nullptr) return fail(TS_ERR_INVALID_ARG, "workspace is NULL (need %zu bytes)", need);
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
    return fail(TS_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(TS_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  return TS_OK;
}

ts_status launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  g_msg[0] = 0;
  return TS_OK;
}

}  // namespace

namespace tsv {

size_t workspace_layout(int64_t batch, int32_t R, int64_t vocab, void* base, Workspace* ws) {
  const size_t rows = (size_t)batch * (size_t)R;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return base ? static_cast<unsigned char*>(base) + at : nullptr;
  };
  Workspace w{};
  w.rowcnt = reinterpret_cast<uint32_t*>(take(rows * 4));
  w.reqcnt = reinterpret_cast<uint32_t*>(take((size_t)batch * 4));
  w.part = reinterpret_cast<Part*>(take(rows * kMaxSplits * sizeof(Part)));
  w.rowres = reinterpret_cast<RowRes*>(take(rows * sizeof(RowRes)));
  w.dpart = reinterpret_cast<DrawPart*>(take((size_t)batch * kMaxSplits * sizeof(DrawPart)));
  w.cmass = reinterpret_cast<uint64_t*>(take(rows * 8 * sizeof(uint64_t)));
  w.best = reinterpret_cast<uint32_t*>(take(rows * 4));
  w.work = reinterpret_cast<uint32_t*>(take(4 * 4));
  w.order = reinterpret_cast<uint32_t*>(take(rows * 4));
  w.creq = reinterpret_cast<uint32_t*>(take((size_t)batch * 4));
  w.slen = reinterpret_cast<int32_t*>(take(rows * 4));
  w.rreq = reinterpret_cast<uint32_t*>(take(rows * 4));
  if (vocab > 0) {
    // sized for fp32 rows, which have the most chunks (at most kMaxSplits)
    int64_t chunk = 0;
    int32_t splits = 0;
    (void)sample_splits(vocab, 4, &splits, &chunk);
    w.cand_splits = splits;
    w.cand = reinterpret_cast<uint64_t*>(
        take(rows * (size_t)splits * (size_t)kSTopK * sizeof(uint64_t)));
  }
  w.bytes = off;
  if (ws) *ws = w;
  return off;
}

}  // namespace tsv

extern "C" {

size_t ts_workspace_size(int64_t batch, int32_t rows_per_req, int64_t vocab) {
  (void)vocab;
  if (batch < 1 || rows_per_req < 1) return 0;
  if (vocab < 1 || vocab > TS_MAX_VOCAB) return 0;
  return tsv::workspace_layout(batch, rows_per_req, vocab, nullptr, nullptr);
}

ts_status ts_workspace_init(void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (!workspace) return fail(TS_ERR_INVALID_ARG, "workspace is NULL");
  return launched(cudaMemsetAsync(workspace, 0, ws_bytes, stream), "cudaMemsetAsync");
}

const char* ts_last_error_message(void) { return g_msg; }

ts_status ts_set_wait_cycles(uint64_t cycles) {
  g_wait_cycles.store(cycles ? cycles : kDefaultWaitCycles, std::memory_order_relaxed);
  g_msg[0] = 0;
  return TS_OK;
}

ts_status ts_device_error(uint32_t* word_host, int clear) {
  if (!word_host) return fail(TS_ERR_INVALID_ARG, "word_host is NULL");
  uint32_t w = 0;
  cudaError_t e = tsv::staged_read_error(&w, clear);
  uint32_t w2 = 0, w3 = 0, w4 = 0;
  if (e == cudaSuccess) e = tsv::row_read_error(&w2, clear);
  if (e == cudaSuccess) e = tsv::softmax_read_error(&w3, clear);
  if (e == cudaSuccess) e = tsv::chain_read_error(&w4, clear);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  w |= (w2 << 8) | (w3 << 16) | (w4 << 24);
  *word_host = w;
  if (w) return fail(TS_ERR_TIMEOUT, "a bounded device wait gave up (word 0x%x)", w);
  g_msg[0] = 0;
  return TS_OK;
}

ts_status ts_softmax_temp(const void* logits, ts_dtype dt, int64_t rows, int64_t vocab,
                          int64_t ld, const float* temperature, float* probs_out,
                          cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if ((st = check_common(rows, vocab, ld)) != TS_OK) return st;
  if (!logits || !probs_out) return fail(TS_ERR_INVALID_ARG, "logits and probs_out are required");
  if (aligned16(logits, ld, dt == TS_BF16 ? 2 : 4))
    return launched(tsv::launch_softmax(logits, dt == TS_BF16, rows, ld, vocab, temperature,
                                        probs_out, stream),
                    "softmax launch");
  if (vocab > tsv::staged_max_vocab(dt == TS_BF16))
    return fail(TS_ERR_INVALID_ARG, "vocab %lld above the staged limit %d", (long long)vocab,
                tsv::staged_max_vocab(dt == TS_BF16));
  tsv::StagedArgs a{};
  a.mode = tsv::kSoftmax;
  a.x = logits;
  a.bf16 = (dt == TS_BF16);
  a.ld = ld;
  a.V = vocab;
  a.rows = rows;
  a.R = 1;
  a.temperature = temperature;
  a.out = probs_out;
  const char* why = "launch";
  return launched(tsv::launch_staged(a, stream, &why), why);
}

ts_status ts_topk_topp_renorm(const float* probs, int64_t rows, int64_t vocab, int64_t ld,
                              const int32_t* top_k, const float* top_p, float* probs_out,
                              cudaStream_t stream) {
  ts_status st;
  if ((st = check_common(rows, vocab, ld)) != TS_OK) return st;
  if (!probs || !probs_out) return fail(TS_ERR_INVALID_ARG, "probs and probs_out are required");
  if (probs_out == probs && ld != vocab)
    return fail(TS_ERR_INVALID_ARG, "in-place renorm needs ld == vocab");
  if (aligned16(probs, ld, 4) && vocab <= tsv::kRowMaxVocab) {
    // the row kernel in its renorm mode: rows streamed through shared memory, no workspace
    tsv::SampleArgs sa{};
    sa.x = probs;
    sa.bf16 = 0;
    sa.ld = ld;
    sa.V = vocab;
    sa.rows = rows;
    sa.R = 1;
    sa.D = 0;
    sa.top_k = top_k;
    sa.top_p = top_p;
    sa.out = probs_out;
    return launched(tsv::launch_renorm_rows(sa, stream), "row renorm launch");
  }
  if (vocab > tsv::staged_max_vocab(0))
    return fail(TS_ERR_INVALID_ARG, "vocab %lld above the staged limit %d", (long long)vocab,
                tsv::staged_max_vocab(0));
  tsv::StagedArgs a{};
  a.mode = tsv::kRenorm;
  a.x = probs;
  a.bf16 = 0;
  a.ld = ld;
  a.V = vocab;
  a.rows = rows;
  a.R = 1;
  a.top_k = top_k;
  a.top_p = top_p;
  a.out = probs_out;
  const char* why = "launch";
  return launched(tsv::launch_staged(a, stream, &why), why);
}

ts_status ts_verify_chain_greedy(const void* target_logits, ts_dtype dt, int64_t batch,
                                 int32_t D, int64_t vocab, int64_t ld,
                                 const int32_t* draft_tokens, int32_t* accepted_tokens,
                                 int32_t* accept_length, int32_t* accept_index,
                                 float* logprobs, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if (D < 0 || D > TS_MAX_DRAFT) return fail(TS_ERR_INVALID_ARG, "D must be in [0, %d]", TS_MAX_DRAFT);
  if ((st = check_common(batch, vocab, ld)) != TS_OK) return st;
  if (!target_logits || !accepted_tokens || !accept_length || (D > 0 && !draft_tokens))
    return fail(TS_ERR_INVALID_ARG, "target_logits, draft_tokens, accepted_tokens and accept_length are required");
  tsv::RowStatArgs a{};
  if ((st = take_workspace(batch, D + 1, vocab, workspace, ws_bytes, &a.ws)) != TS_OK) return st;
  a.x = target_logits;
  a.ld = ld;
  a.V = vocab;
  a.rows = batch * (D + 1);
  choose_splits(a.rows, vocab, 2048, &a.splits, &a.split_len);
  a.vec = aligned16(target_logits, ld, dt == TS_BF16 ? 2 : 4);
  a.want_lse = logprobs != nullptr;
  a.kind = 0;
  a.D = D;
  a.draft_tokens = draft_tokens;
  a.accepted_tokens = accepted_tokens;
  a.accept_length = accept_length;
  a.accept_index = accept_index;
  a.logprobs = logprobs;
  return launched(tsv::launch_rowstat(a, dt == TS_BF16, stream), "greedy verify launch");
}

ts_status ts_verify_chain_greedy_ragged(const void* target_logits, ts_dtype dt, int64_t batch,
                                        int32_t D, int64_t vocab, int64_t ld,
                                        const int32_t* qo_indptr, int64_t total_rows,
                                        const int32_t* draft_tokens, int32_t* accepted_tokens,
                                        int32_t* accept_length, int32_t* accept_index,
                                        float* logprobs, void* workspace, size_t ws_bytes,
                                        cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if (D < 0 || D > TS_MAX_DRAFT) return fail(TS_ERR_INVALID_ARG, "D must be in [0, %d]", TS_MAX_DRAFT);
  if ((st = check_common(batch, vocab, ld)) != TS_OK) return st;
  const int32_t R = D + 1;
  if (!target_logits || !qo_indptr || !accepted_tokens || !accept_length || (D > 0 && !draft_tokens))
    return fail(TS_ERR_INVALID_ARG,
                "target_logits, qo_indptr, draft_tokens, accepted_tokens and accept_length are required");
  if (total_rows < 1 || total_rows > batch * (int64_t)R)
    return fail(TS_ERR_INVALID_ARG, "total_rows must be in [1, batch * (D + 1)]");
  tsv::RowStatArgs a{};
  if ((st = take_workspace(batch, R, vocab, workspace, ws_bytes, &a.ws)) != TS_OK) return st;
  // outputs of a window that does not fit: accept_length 0, tokens and indices -1,
  // logprobs 0 (the others are overwritten)
  const size_t outs = (size_t)batch * (size_t)R * sizeof(int32_t);
  cudaError_t e = cudaMemsetAsync(accept_length, 0, (size_t)batch * sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(accepted_tokens, 0xFF, outs, stream);
  if (e == cudaSuccess && accept_index) e = cudaMemsetAsync(accept_index, 0xFF, outs, stream);
  if (e == cudaSuccess && logprobs) e = cudaMemsetAsync(logprobs, 0, outs, stream);
  if (e != cudaSuccess) return launched(e, "ragged greedy verify clear");
  a.x = target_logits;
  a.ld = ld;
  a.V = vocab;
  a.rows = total_rows;
  choose_splits(a.rows, vocab, 2048, &a.splits, &a.split_len);
  a.vec = aligned16(target_logits, ld, dt == TS_BF16 ? 2 : 4);
  a.want_lse = logprobs != nullptr;
  a.kind = 0;
  a.D = D;
  a.draft_tokens = draft_tokens;
  a.accepted_tokens = accepted_tokens;
  a.accept_length = accept_length;
  a.accept_index = accept_index;
  a.logprobs = logprobs;
  a.qo = qo_indptr;
  a.nreq = batch;
  return launched(tsv::launch_rowstat(a, dt == TS_BF16, stream), "ragged greedy verify launch");
}

ts_status ts_chain_spec_sampling(const ts_chain_args* p, void* workspace, size_t ws_bytes,
                                 cudaStream_t stream) {
  if (!p) return fail(TS_ERR_INVALID_ARG, "args is NULL");
  ts_status st;
  if ((st = check_dtype(p->target_dtype)) != TS_OK) return st;
  if (p->D < 0 || p->D > TS_MAX_DRAFT) return fail(TS_ERR_INVALID_ARG, "D must be in [0, %d]", TS_MAX_DRAFT);
  if ((st = check_common(p->batch, p->vocab, p->ld)) != TS_OK) return st;
  if (!p->target || !p->accepted_tokens || !p->accept_length || (p->D > 0 && !p->draft_tokens))
    return fail(TS_ERR_INVALID_ARG, "target, draft_tokens, accepted_tokens and accept_length are required");
  if (!p->uniforms && (!p->seed || !p->offset))
    return fail(TS_ERR_INVALID_ARG, "seed and offset are required when uniforms is NULL");
  if (p->draft_probs && p->ld_draft < p->vocab)
    return fail(TS_ERR_INVALID_ARG, "ld_draft must be >= vocab");
  const int32_t R = p->D + 1;
  const float thr_s = unit_threshold(p->threshold_single), thr_a = unit_threshold(p->threshold_acc);
  const bool relaxed = thr_s < 1.f || thr_a < 1.f;
  if (relaxed && p->draft_probs)
    return fail(TS_ERR_INVALID_ARG, "relaxed acceptance thresholds are target-only");
  const bool ragged = p->qo_indptr != nullptr;
  if (ragged && (p->total_rows < 1 || p->total_rows > p->batch * (int64_t)R))
    return fail(TS_ERR_INVALID_ARG, "total_rows must be in [1, batch * (D + 1)]");
  const bool next_knobs = relaxed || p->min_p != nullptr || ragged;
  if (next_knobs && !p->target_is_logits)
    return fail(TS_ERR_INVALID_ARG,
                "min_p, relaxed thresholds and ragged batches need logit targets");
  if (!p->target_is_logits) {
    if (p->target_dtype != TS_F32)
      return fail(TS_ERR_UNSUPPORTED_DTYPE, "probability targets must be fp32");
    tsv::DrawArgs a{};
    if ((st = take_workspace(p->batch, R, p->vocab, workspace, ws_bytes, &a.ws)) != TS_OK) return st;
    a.p = static_cast<const float*>(p->target);
    a.ld = p->ld;
    a.V = p->vocab;
    a.B = p->batch;
    a.D = p->D;
    a.q = p->draft_probs;
    a.ld_q = p->ld_draft;
    a.drafts = p->draft_tokens;
    a.seed = p->seed;
    a.offset = p->offset;
    a.uniforms = p->uniforms;
    choose_splits(p->batch, p->vocab, 4096, &a.splits, &a.split_len);
    a.vec = aligned16(p->target, p->ld, 4) && (!p->draft_probs || aligned16(p->draft_probs, p->ld_draft, 4));
    a.accepted_tokens = p->accepted_tokens;
    a.accept_length = p->accept_length;
    a.accept_index = p->accept_index;
    a.logprobs = p->logprobs;
    return launched(tsv::launch_draw_probs(a, stream), "probability-row chain launch");
  }
  if (p->vocab > tsv::staged_max_vocab(p->target_dtype == TS_BF16))
    return fail(TS_ERR_INVALID_ARG, "vocab %lld above the staged limit %d", (long long)p->vocab,
                tsv::staged_max_vocab(p->target_dtype == TS_BF16));
  tsv::StagedArgs a{};
  if ((st = take_workspace(p->batch, R, p->vocab, workspace, ws_bytes, &a.ws)) != TS_OK) return st;
  a.mode = tsv::kChain;
  a.x = p->target;
  a.bf16 = (p->target_dtype == TS_BF16);
  a.ld = p->ld;
  a.V = p->vocab;
  a.rows = p->batch * R;
  a.R = R;
  a.D = p->D;
  a.temperature = p->temperature;
  a.top_k = p->top_k;
  a.top_p = p->top_p;
  a.draft_tokens = p->draft_tokens;
  a.seed = p->seed;
  a.offset = p->offset;
  a.uniforms = p->uniforms;
  a.accepted_tokens = p->accepted_tokens;
  a.accept_length = p->accept_length;
  a.accept_index = p->accept_index;
  a.logprobs = p->logprobs;
  const int esize = p->target_dtype == TS_BF16 ? 2 : 4;
  tsv::SampleArgs sa{};
  if (aligned16(p->target, p->ld, esize) && p->vocab <= tsv::kRowMaxVocab &&
      tsv::sample_splits(p->vocab, esize, &sa.splits, &sa.chunk) && sa.splits <= a.ws.cand_splits) {
    // Every row: the row-streaming kernel.
    sa.x = p->target;
    sa.bf16 = a.bf16;
    sa.ld = p->ld;
    sa.V = p->vocab;
    sa.rows = a.rows;
    sa.R = R;
    sa.D = p->D;
    sa.temperature = p->temperature;
    sa.top_k = p->top_k;
    sa.top_p = p->top_p;
    sa.draft_tokens = p->draft_tokens;
    sa.seed = p->seed;
    sa.offset = p->offset;
    sa.uniforms = p->uniforms;
    sa.accepted_tokens = p->accepted_tokens;
    sa.accept_length = p->accept_length;
    sa.accept_index = p->accept_index;
    sa.logprobs = p->logprobs;
    sa.ws = a.ws;
    sa.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
    sa.q = p->draft_probs;
    sa.ld_q = p->ld_draft;
    sa.min_p = p->min_p;
    sa.thr_single = thr_s;
    sa.thr_acc = thr_a;
    sa.nreq = p->batch;
    if (ragged) {
      sa.qo = p->qo_indptr;
      sa.rows = p->total_rows;
    }
    return launched(tsv::launch_chain(sa, stream), "row-streaming chain launch");
  }
  if (next_knobs)
    return fail(TS_ERR_INVALID_ARG,
                "min_p, relaxed thresholds and ragged batches need 16-byte aligned rows and "
                "vocab <= %lld",
                (long long)tsv::kRowMaxVocab);
  if (p->draft_probs)
    return fail(TS_ERR_INVALID_ARG,
                "logit targets with draft probabilities need 16-byte aligned rows and vocab "
                "<= %lld",
                (long long)tsv::kRowMaxVocab);
  if (p->temperature) {
    // Greedy requests need only the argmax of each row: a streaming pass handles them,
    // and the staged kernel skips them.
    tsv::RowStatArgs g{};
    g.ws = a.ws;
    g.x = p->target;
    g.ld = p->ld;
    g.V = p->vocab;
    g.rows = a.rows;
    choose_splits(g.rows, p->vocab, 2048, &g.splits, &g.split_len);
    g.vec = aligned16(p->target, p->ld, esize);
    g.want_lse = p->logprobs != nullptr;
    g.kind = 0;
    g.D = p->D;
    g.draft_tokens = p->draft_tokens;
    g.accepted_tokens = p->accepted_tokens;
    g.accept_length = p->accept_length;
    g.accept_index = p->accept_index;
    g.logprobs = p->logprobs;
    g.req_temperature = p->temperature;
    cudaError_t e = tsv::launch_rowstat(g, p->target_dtype == TS_BF16, stream);
    if (e != cudaSuccess) return cuda_fail(e, "greedy rows launch");
    a.skip_greedy = 1;
  }
  const char* why = "target-only chain launch";
  return launched(tsv::launch_staged(a, stream, &why), why);
}

ts_status ts_sample_from_logits(const ts_sample_args* p, void* workspace, size_t ws_bytes,
                                cudaStream_t stream) {
  if (!p) return fail(TS_ERR_INVALID_ARG, "args is NULL");
  ts_status st;
  if ((st = check_dtype(p->dtype)) != TS_OK) return st;
  if (p->n_per_req < 1) return fail(TS_ERR_INVALID_ARG, "n_per_req must be >= 1");
  if (p->batch < 1) return fail(TS_ERR_INVALID_ARG, "batch must be >= 1");
  const int64_t rows = p->batch * (int64_t)p->n_per_req;
  if ((st = check_common(rows, p->vocab, p->ld)) != TS_OK) return st;
  if (!p->logits || !p->tokens) return fail(TS_ERR_INVALID_ARG, "logits and tokens are required");
  if (!p->uniforms && (!p->seed || !p->offset))
    return fail(TS_ERR_INVALID_ARG, "seed and offset are required when uniforms is NULL");
  if (p->filter_order != TS_FILTER_TOP_K_FIRST && p->filter_order != TS_FILTER_JOINT)
    return fail(TS_ERR_INVALID_ARG, "filter_order must be TS_FILTER_TOP_K_FIRST or TS_FILTER_JOINT");
  if (p->probs && p->ld_probs < p->vocab) return fail(TS_ERR_INVALID_ARG, "ld_probs must be >= vocab");
  const int esize = p->dtype == TS_BF16 ? 2 : 4;
  tsv::SampleArgs sa{};
  if (!aligned16(p->logits, p->ld, esize) || p->vocab > tsv::kRowMaxVocab ||
      !tsv::sample_splits(p->vocab, esize, &sa.splits, &sa.chunk))
    return fail(TS_ERR_INVALID_ARG, "sampling needs 16-byte aligned rows and vocab <= %lld",
                (long long)tsv::kRowMaxVocab);
  if ((st = take_workspace(rows, 1, p->vocab, workspace, ws_bytes, &sa.ws)) != TS_OK) return st;
  if (sa.splits > sa.ws.cand_splits)
    return fail(TS_ERR_INVALID_ARG, "vocab %lld needs more row chunks than the workspace holds",
                (long long)p->vocab);
  sa.x = p->logits;
  sa.bf16 = p->dtype == TS_BF16;
  sa.ld = p->ld;
  sa.V = p->vocab;
  sa.rows = rows;
  sa.R = 1;
  sa.D = 0;
  sa.temperature = p->temperature;
  sa.top_k = p->top_k;
  sa.top_p = p->top_p;
  sa.min_p = p->min_p;
  sa.joint = p->filter_order == TS_FILTER_JOINT;
  sa.thr_single = 1.f;
  sa.thr_acc = 1.f;
  sa.sample_n = p->n_per_req;
  sa.seed = p->seed;
  sa.offset = p->offset;
  sa.uniforms = p->uniforms;
  sa.accepted_tokens = p->tokens;
  sa.accept_length = sa.ws.slen;
  sa.logprobs = p->logprobs;
  sa.probs_out = p->probs;
  sa.ld_probs = p->ld_probs;
  sa.probs_row = p->probs_row;
  sa.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
  sa.nreq = rows;
  return launched(tsv::launch_chain(sa, stream), "sampling launch");
}

ts_status ts_gumbel_max_sample(const void* logits, ts_dtype dt, int64_t batch,
                               int32_t n_per_req, int64_t vocab, int64_t ld,
                               const float* temperature, const int64_t* seed,
                               const int64_t* offset, int32_t* tokens_out, void* workspace,
                               size_t ws_bytes, cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if (n_per_req < 1) return fail(TS_ERR_INVALID_ARG, "n_per_req must be >= 1");
  if ((st = check_common(batch * (int64_t)n_per_req, vocab, ld)) != TS_OK) return st;
  if (!logits || !temperature || !seed || !offset || !tokens_out)
    return fail(TS_ERR_INVALID_ARG, "logits, temperature, seed, offset and tokens_out are required");
  tsv::Workspace ws{};
  if ((st = take_workspace(batch, n_per_req, vocab, workspace, ws_bytes, &ws)) != TS_OK) return st;
  const int esize = dt == TS_BF16 ? 2 : 4;
  if (aligned16(logits, ld, esize)) {
    // a chunk is one warp's claim: 128 to 1024 vectors, about two a warp over the whole
    // call, and no more than kMaxSplits a row
    tsv::GumbelArgs g{};
    const int64_t rows = batch * n_per_req;
    const int64_t nv = vocab / (16 / esize);
    const int64_t ctas = (int64_t)sm_count() * tsv::gumbel_ctas_per_sm(dt == TS_BF16);
    int64_t cv = (rows * nv + 2 * 8 * ctas - 1) / (2 * 8 * ctas);
    cv = std::min<int64_t>(std::max<int64_t>(cv, 128), 1024);
    cv = std::max<int64_t>(cv, (nv + tsv::kMaxSplits - 1) / tsv::kMaxSplits);
    const int64_t cpr = std::max<int64_t>(1, (nv + cv - 1) / cv);
    g.x = logits;
    g.ld = ld;
    g.V = vocab;
    g.rows = rows;
    g.n_per_req = n_per_req;
    g.temperature = temperature;
    g.seed = seed;
    g.offset = offset;
    g.tokens_out = tokens_out;
    g.chunk_vecs = cv;
    g.cpr = (int32_t)cpr;
    g.total_chunks = (uint32_t)(rows * cpr);
    g.grid = (int32_t)std::min<int64_t>(ctas, (rows * cpr + 7) / 8);
    g.ws = ws;
    return launched(tsv::launch_gumbel(g, dt == TS_BF16, stream), "Gumbel launch");
  }
  tsv::RowStatArgs a{};
  a.ws = ws;
  a.x = logits;
  a.ld = ld;
  a.V = vocab;
  a.rows = batch * n_per_req;
  choose_splits(a.rows, vocab, 2048, &a.splits, &a.split_len);
  a.vec = 0;
  a.kind = 2;
  a.temperature = temperature;
  a.seed = seed;
  a.offset = offset;
  a.n_per_req = n_per_req;
  a.tokens_out = tokens_out;
  return launched(tsv::launch_rowstat(a, dt == TS_BF16, stream), "Gumbel launch");
}

ts_status ts_gather_logprobs(const void* x, ts_dtype dt, int32_t is_probs, int64_t rows,
                             int64_t vocab, int64_t ld, const int32_t* tokens, float* out,
                             void* workspace, size_t ws_bytes, cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if ((st = check_common(rows, vocab, ld)) != TS_OK) return st;
  if (!x || !tokens || !out) return fail(TS_ERR_INVALID_ARG, "x, tokens and out are required");
  if (is_probs) {
    if (dt != TS_F32) return fail(TS_ERR_UNSUPPORTED_DTYPE, "probabilities must be fp32");
    return launched(tsv::launch_logprobs_probs(static_cast<const float*>(x), ld, vocab, rows,
                                               tokens, out, stream),
                    "logprobs launch");
  }
  tsv::RowStatArgs a{};
  if ((st = take_workspace(rows, 1, vocab, workspace, ws_bytes, &a.ws)) != TS_OK) return st;
  a.x = x;
  a.ld = ld;
  a.V = vocab;
  a.rows = rows;
  choose_splits(rows, vocab, 2048, &a.splits, &a.split_len);
  a.vec = aligned16(x, ld, dt == TS_BF16 ? 2 : 4);
  a.want_lse = 1;
  a.kind = 1;
  a.lp_tokens = tokens;
  a.lp_out = out;
  return launched(tsv::launch_rowstat(a, dt == TS_BF16, stream), "logprobs launch");
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Greedy chain verification without a caller workspace.
//
// Some callers cannot hand the library device memory: a host that binds the C ABI
// without any device allocator of its own, or code whose device memory is a fixed budget
// owned by another allocator that the library may not draw from. For them this variant
// keeps its scratch
// (arrival counters and per-split partials) in a file-scope device array that every GPU
// loading the library holds until the process exits. Its size is fixed, so the number
// of rows it can serve is capped.

namespace {

constexpr size_t kStaticScratchBytes = (size_t)4 << 20;  // 4 MiB per device
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The device address of the scratch array on the current device. (In host code the
// array's name is only a host-side handle, never a device pointer.) Looked up on every
// call: the lookup allocates nothing and launches nothing, and a cached address could
// outlive the context it was taken in (after cudaDeviceReset, say). The first lookup on
// a device loads the library's device code there.
ts_status static_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  *out = p;
  return TS_OK;
}

}  // namespace

extern "C" ts_status ts_verify_chain_greedy_static(const void* target_logits, ts_dtype dt,
                                                   int64_t batch, int32_t D, int64_t vocab,
                                                   int64_t ld, const int32_t* draft_tokens,
                                                   int32_t* accepted_tokens,
                                                   int32_t* accept_length,
                                                   int32_t* accept_index, float* logprobs,
                                                   cudaStream_t stream) {
  ts_status st;
  if ((st = check_dtype(dt)) != TS_OK) return st;
  if (D < 0 || D > TS_MAX_DRAFT) return fail(TS_ERR_INVALID_ARG, "D must be in [0, %d]", TS_MAX_DRAFT);
  if ((st = check_common(batch, vocab, ld)) != TS_OK) return st;
  if (!target_logits || !accepted_tokens || !accept_length || (D > 0 && !draft_tokens))
    return fail(TS_ERR_INVALID_ARG, "target_logits, draft_tokens, accepted_tokens and accept_length are required");
  const int64_t rows = batch * (D + 1);
  if (rows > TS_STATIC_MAX_ROWS)
    return fail(TS_ERR_INVALID_ARG,
                "batch*(D+1) = %lld rows exceeds the static scratch limit of %d rows",
                (long long)rows, TS_STATIC_MAX_ROWS);
  if (tsv::workspace_layout(batch, D + 1, 0, nullptr, nullptr) > kStaticScratchBytes)
    return fail(TS_ERR_INVALID_ARG, "the call needs more than the %zu-byte static scratch",
                kStaticScratchBytes);
  void* base = nullptr;
  if ((st = static_scratch(&base)) != TS_OK) return st;
  tsv::RowStatArgs a{};
  tsv::workspace_layout(batch, D + 1, 0, base, &a.ws);
  // The array keeps whatever the previous call left; the arrival counters must start at 0.
  cudaError_t e = cudaMemsetAsync(a.ws.rowcnt, 0, (size_t)rows * sizeof(uint32_t), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(a.ws.reqcnt, 0, (size_t)batch * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the static scratch counters");
  a.x = target_logits;
  a.ld = ld;
  a.V = vocab;
  a.rows = rows;
  choose_splits(a.rows, vocab, 2048, &a.splits, &a.split_len);
  a.vec = aligned16(target_logits, ld, dt == TS_BF16 ? 2 : 4);
  a.want_lse = logprobs != nullptr;
  a.kind = 0;
  a.D = D;
  a.draft_tokens = draft_tokens;
  a.accepted_tokens = accepted_tokens;
  a.accept_length = accept_length;
  a.accept_index = accept_index;
  a.logprobs = logprobs;
  return launched(tsv::launch_rowstat(a, dt == TS_BF16, stream), "greedy verify (static scratch) launch");
}
