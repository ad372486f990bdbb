/*
 * sdv.h -- speculative-decoding verify path on one GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels for the draft -> verify -> accept ->
 * commit/rewind transaction of greedy speculative decoding on a dense
 * decoder with a paged KV cache. Plain pointers and sizes only.
 *
 * Sources, by page title and section:
 *   [TS] TensorSharp, "Speculative decoding": the shared loop / trunk seam
 *        (SpecForward, SpecEnsureCapacity, SpecRewindCache, CacheSeqLen);
 *        the protocol (draft, verify, rollback, commit); n-gram lookup.
 *   [PI] pegainfer, "Qwen3 DFlash speculative decoding": the transaction
 *        (propose, verify, accept_greedy, commit/LIFO drop); draft-seed
 *        alignment; capture-shape gotcha (span truncation, KV length read
 *        at run time); context limit (reject cleanly).
 *   [CA] CoreAI model zoo, "spec-decode n-gram on a dense target": dense
 *        rollback by position; adaptive K; argmax the rows in place.
 *
 * Conventions for every call:
 *   - Pointers named d_* are device pointers; h_* are host pointers. All
 *     device buffers are allocated by the caller and borrowed: the library
 *     never allocates device memory and never frees what it is given. They
 *     must stay valid for the life of the context.
 *   - `stream` is a cudaStream_t. Every call that takes one only enqueues
 *     work on it and returns; nothing synchronises unless stated.
 *   - Return value: SDV_OK (0) or a negative SDV_ERR_* code. Argument errors
 *     found on the host return at once and enqueue nothing. Errors found on
 *     the device (a token id >= vocab, a span longer than declared, a page
 *     table without room, a rewind past the written length, the pool out of
 *     pages) set a device status word; kernels then skip any memory access
 *     the error would make unsafe, and sdv_get_status reports the first
 *     such error. No exception crosses this boundary.
 *   - Weights are bf16, row-major W[out][in], 16-byte aligned; norm gains
 *     are bf16 vectors. Activations are bf16 with fp32 accumulation and an
 *     fp32 residual stream.
 *   - A batch is B sequences, B <= max_batch; sequence b of a call is
 *     sequence slot b of the context. Spans are packed: rows
 *     row_off[b] .. row_off[b+1]-1 belong to sequence b (row_off[0] = 0,
 *     row_off[B] = R, the total rows). A sequence with an empty span is left
 *     untouched.
 */
#ifndef SDV_H
#define SDV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SDV_OK 0
#define SDV_ERR_ARG (-1)            /* invalid argument (host) or invalid span/rewind (device) */
#define SDV_ERR_CAPACITY (-2)       /* out of pages, or past the page table / max_context */
#define SDV_ERR_CUDA (-3)           /* a CUDA runtime call failed */
#define SDV_ERR_DEVICE (-4)         /* bad device input: a token id outside [0, vocab), a bad page id */
#define SDV_ERR_DEVICE_TIMEOUT (-5) /* a bounded device wait gave up */
#define SDV_ERR_UNSUPPORTED (-6)    /* a shape this build does not handle */

typedef struct sdv_ctx sdv_ctx; /* opaque; owns only host-side state */

/* Decoder shape. head_dim must be 64 or 128; hidden, n_q_heads*head_dim and
 * ffn must be multiples of 8 (16-byte rows). */
typedef struct {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    float rms_eps, rope_theta;
    int qk_norm; /* 1: per-head RMSNorm on q and k before RoPE */
    /* [TS] sliding-window caches: with swa_window > 0, layer l is a local layer
     * (its row at position q attends positions q - swa_window + 1 .. q) unless
     * swa_global_every > 0 and (l + 1) % swa_global_every == 0. A local layer
     * keeps exactly one window of positions in a ring (position p in slot
     * p % swa_window, on the sequence's first swa_window / page_size pages).
     * swa_window must be a multiple of page_size and at least max_span. */
    int swa_window, swa_global_every;
} sdv_model_cfg;

/* Cache and call limits. Attention takes its TMA-fed path when page_size is
 * a power of two in [8, 128] and n_kv_heads <= 16; otherwise a slower kernel
 * that loads pages with ordinary loads serves the same calls. */
typedef struct {
    int page_size;      /* tokens per KV page (16) */
    int n_pages;        /* pages in the pool */
    int max_batch;      /* sequence slots */
    int max_rows;       /* rows per sdv_spec_forward call, <= 128 */
    int max_span;       /* rows per sequence per call, <= max_rows */
    int max_context;    /* tokens per sequence; page table = ceil(max_context/page_size) slots */
    int ngram_capacity; /* history tokens kept per sequence for n-gram lookup (0: none); needs vocab <= 2^21 */
    int ngram_max_order; /* n-gram orders indexed per sequence, 1..6 (0: 2) */
} sdv_cache_cfg;

typedef struct {
    const void *attn_norm;  /* [hidden] */
    const void *wq;         /* [n_q_heads*head_dim][hidden] */
    const void *wk;         /* [n_kv_heads*head_dim][hidden] */
    const void *wv;         /* [n_kv_heads*head_dim][hidden] */
    const void *q_norm;     /* [head_dim] */
    const void *k_norm;     /* [head_dim] */
    const void *wo;         /* [hidden][n_q_heads*head_dim] */
    const void *ffn_norm;   /* [hidden] */
    const void *w_gate;     /* [ffn][hidden] */
    const void *w_up;       /* [ffn][hidden] */
    const void *w_down;     /* [hidden][ffn] */
} sdv_layer_weights;

typedef struct {
    const void *embed;              /* [vocab][hidden] */
    const void *lm_head;            /* [vocab][hidden] (untied) */
    const void *final_norm;         /* [hidden] */
    const sdv_layer_weights *layers; /* host array of n_layers entries (copied at create) */
} sdv_weights;

/* Bytes of the caller-owned workspace (scratch, the device status word, page
 * tables, lengths, the n-gram index and loop state). Allocate with 256-byte
 * alignment; the library zero-initialises what it needs in sdv_create. The
 * size depends on the configuration and on the current device's SM count (the
 * attention's work layout), so ask on the device the context will use. */
int sdv_workspace_bytes(const sdv_model_cfg *m, const sdv_cache_cfg *c, size_t *bytes);

/* Bytes of the caller-owned KV pool. Layout (bf16):
 *   pool[layer][page][kv (0 = K, 1 = V)][kv_head][slot (page_size)][head_dim]
 * Token at position p of sequence b lives in page table[b][p / page_size],
 * slot p % page_size. K is stored after head RMSNorm and RoPE. */
int sdv_kv_pool_bytes(const sdv_model_cfg *m, const sdv_cache_cfg *c, size_t *bytes);

/* Create a context on the current CUDA device. Builds TMA descriptors for the
 * weights and activation buffers, the RoPE table, the empty page pool (every
 * page free; the first reservation takes page 0), zero lengths and an empty
 * n-gram index, enqueued on `stream`. The weights, pool and workspace are
 * borrowed. Returns SDV_ERR_UNSUPPORTED on a device without sm_103a-class
 * tcgen05 or on an unsupported shape. */
int sdv_create(const sdv_model_cfg *m, const sdv_cache_cfg *c, const sdv_weights *w, void *d_kv_pool,
               void *d_workspace, void *stream, sdv_ctx **out);

/* Free the library's host state (never the borrowed device buffers). */
int sdv_destroy(sdv_ctx *ctx);

/* [TS] SpecEnsureCapacity; [PI] context limit.
 * Reserve pages so sequence b holds d_required[b] tokens (d_required[b] < 0:
 * leave b alone). Sequences are served in order b = 0..B-1, each filling its
 * empty page-table slots in ascending order from the top of the free stack.
 * All-or-nothing: if any sequence would pass its page table or the pool runs
 * dry, nothing changes and the device status becomes SDV_ERR_CAPACITY. */
int sdv_ensure_capacity(sdv_ctx *ctx, const int32_t *d_required, int B, void *stream);

/* [PI] the transaction, Verify; [TS] SpecForward; [CA] dense rollback.
 * One forward over each sequence's span, rows at positions L_b .. L_b+S_b-1
 * where L_b is the cache length before the call; every row's K/V is written
 * at its true position before any row attends, each row attends positions
 * 0..its own, and afterwards L_b += S_b. The cache must already hold room
 * (sdv_ensure_capacity); a span past it, S_b > max_span or R > max_rows sets
 * the device status.
 *   d_tokens   [R] int32 token ids; row 0 of a span is the sequence's current
 *              token, then its drafts.
 *   d_row_off  [B+1] int32, device-resident, so one launch shape (fixed by
 *              max_rows / max_span) serves any mix of span lengths.
 *   max_rows   host bound on R (<= cfg max_rows); sets the GEMM width.
 *   max_span   host bound on every S_b (<= cfg max_span).
 *   d_argmax   [R] int32 out: per-row argmax of the logits, lowest index on
 *              an exact tie. Only rows < R are written.
 *   d_logits   [R][vocab] fp32 out, or NULL. When NULL no logits are stored
 *              anywhere: the argmax is reduced inside the LM-head kernel. */
int sdv_spec_forward(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, int B, int max_rows,
                     int max_span, int32_t *d_argmax, float *d_logits, void *stream);

/* [TS] the protocol, Verify: "the caller's sampler draws each row and drafts
 * are accepted while the drawn token matches".
 * The same forward as sdv_spec_forward, with each row drawn from
 * softmax(logits / T_b) instead of taking its argmax: row r of sequence b at
 * position p draws argmax_v(logit_v / T_b + g_v), g_v = -log(-log u_v) (the
 * Gumbel-max construction), in float32. u_v comes from SplitMix64 streams
 * (Steele, Lea and Flood 2014; stream(k)[i] = mix64(k + (i+1) *
 * 0x9E3779B97F4A7C15)): x = stream(stream(stream(seed)[b])[p])[v],
 * u = ((x >> 41) + 1/2) * 2^-23. The noise of a position depends only on
 * (seed, b, p, v), so with a fixed seed a position draws the same token
 * whether it is verified in a span or decoded alone, and sdv_accept_greedy
 * on the drawn tokens is the sampled accept rule (speculation stays lossless).
 *   d_temperature [B] float (device): T_b; T_b <= 0 draws the argmax (greedy).
 *   seed          the generation's key; keep it fixed across a generation.
 *   d_drawn       [R] int32 out: the drawn token of each row.
 *   d_logits      as in sdv_spec_forward (the unperturbed logits), or NULL.
 * Other arguments, errors and effects as sdv_spec_forward; a NULL
 * d_temperature returns SDV_ERR_ARG. */
int sdv_spec_forward_sampled(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, int B, int max_rows,
                             int max_span, const float *d_temperature, uint64_t seed, int32_t *d_drawn,
                             float *d_logits, void *stream);

/* [PI] the transaction, Accept; draft-seed alignment; [TS] the protocol.
 * For each sequence with S_b = k+1 >= 1 rows (drafts d_1..d_k = span rows
 * 1..k, argmax a_0..a_k): m_b = the largest j <= k with d_i == a_{i-1} for
 * all i <= j. Writes d_n_accept[b] = m_b, d_committed[b*max_commit + i] =
 * a_i for i <= m_b, d_n_commit[b] = m_b + 1, and d_new_len[b] =
 * (L_b - S_b) + m_b + 1 with L_b the length after the forward. A sequence
 * with an empty span gets m = -1, n_commit = 0 and new_len = -1 (pass it to
 * sdv_rewind_cache unchanged: -1 means leave alone). The loop state of
 * sdv_gen_init (current token, tokens generated, adaptive K) advances too.
 * max_commit >= max_span. */
int sdv_accept_greedy(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, const int32_t *d_argmax,
                      int B, int max_commit, int32_t *d_n_accept, int32_t *d_committed, int32_t *d_n_commit,
                      int32_t *d_new_len, void *stream);

/* [TS] SpecRewindCache; [PI] LIFO drop; [CA] rollback == do not advance.
 * Set each length to d_length[b] (< 0: leave b alone), which must not pass
 * the written length (else SDV_ERR_ARG in the device status, nothing
 * changes). Rows past it stay in the pages as stale data that nothing reads.
 * Pages past ceil(length / page_size) go back to the free stack for
 * b = B-1 down to 0, highest slot first, so a rewind to the lengths before an
 * sdv_ensure_capacity restores the pool exactly.
 * Sliding-window layers ([TS] sliding-window caches and rollback): the last
 * forward kept what its rows evicted from each local layer's ring; rows of
 * that forward at or past the new length are rejected, and their slots get
 * back the positions they held (a full acceptance restores nothing). A rewind
 * below the start of the last forward's span, once a ring has wrapped, would
 * need positions no longer kept: SDV_ERR_ARG, nothing changes. */
int sdv_rewind_cache(sdv_ctx *ctx, const int32_t *d_length, int B, void *stream);

/* [TS] CacheSeqLen: copy the max_batch cache lengths into d_len. */
int sdv_cache_seq_len(sdv_ctx *ctx, int32_t *d_len, void *stream);

/* Copy the page tables (d_table[max_batch][pages_per_seq], unused slots -1),
 * the pages held per sequence (d_n_pages[max_batch]) and the free-stack
 * depth (d_free_top[1]) for inspection. */
int sdv_page_table(sdv_ctx *ctx, int32_t *d_table, int32_t *d_n_pages, int32_t *d_free_top, void *stream);

/* [TS] n-gram: append d_counts[b] tokens (d_tokens[b*stride + i]) to sequence
 * b's history; each new token at position p completes the contexts of the
 * n tokens before it (n = 1..ngram_max_order), and each such context -> p
 * goes into that order's hash index of the sequence ([TS]: one incrementally
 * maintained index per n-gram order; exact keys; a later insertion of the
 * same context overwrites, so lookup returns the most recent occurrence). A
 * token outside [0, 2^21) sets SDV_ERR_DEVICE and stops the append. */
int sdv_ngram_commit(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_counts, int B, int stride,
                     void *stream);

/* Loop state for the proposers: sequence b's current token d_first[b] (the
 * argmax of its prompt's last row), 1 token generated, a budget of
 * d_budget[b] generated tokens, draft length k_init, and whether K adapts.
 * [CA] adaptive K: start at 1; +2 after a fully accepted round; -1 after any
 * rejection; clamp to [1, k_max]; a round without drafts keeps K. */
int sdv_gen_init(sdv_ctx *ctx, const int32_t *d_first, const int32_t *d_budget, int B, int k_init, int adaptive,
                 int k_max, void *stream);

/* [CA] --ngram-min; [TS] --spec-pmin (for the n-gram drafter it scales the
 * required match length). The n-gram drafter proposes off the longest
 * context of n tokens, n_req <= n <= ngram_max_order, that occurred earlier in
 * the history with a follower, where n_req = min_order + floor(pmin *
 * (ngram_max_order - min_order) + 1/2). Defaults: min_order 2, pmin 0.
 * min_order in [1, ngram_max_order], pmin in [0, 1], else SDV_ERR_ARG. Host
 * state, read when sdv_propose is enqueued (so a captured graph keeps the
 * values it was captured with). */
int sdv_ngram_params(sdv_ctx *ctx, int min_order, float pmin);

#define SDV_DRAFT_NONE 0  /* plain one-row steps (speculation off) */
#define SDV_DRAFT_NGRAM 1 /* n-gram prompt lookup over the sequence's history (sdv_ngram_params) */
#define SDV_DRAFT_TABLE 2 /* drafts read from d_table[b*table_stride + g], g = tokens generated so far */

/* Build the next verify span of every sequence from the loop state:
 * [current, d_1..d_k] with k = min(K_b, budget_b - generated_b - 1) drafts at
 * most ([PI] capture-shape gotcha: the span is cut to the output budget), or
 * an empty span once the budget is met. Writes d_tokens (packed, capacity
 * B*max_span), d_row_off [B+1] and d_required[b] = L_b + S_b (or -1) for
 * sdv_ensure_capacity. Spans longer than max_span are cut to it. */
int sdv_propose(sdv_ctx *ctx, int drafter, const int32_t *d_table, int table_stride, int B, int max_span,
                int32_t *d_tokens, int32_t *d_row_off, int32_t *d_required, void *stream);

/* [TS] Reset: empty sequence b's cache (all its pages return to the pool),
 * n-gram history and loop state. */
int sdv_reset_seq(sdv_ctx *ctx, int b, void *stream);

/* Synchronise the device, copy the status word to *h_status and clear it. */
int sdv_get_status(sdv_ctx *ctx, int32_t *h_status);

/* A static string naming an SDV_* code. */
const char *sdv_status_str(int code);

/* Op-level call for parity checks at full size: paged attention of layer
 * `layer` for the query rows d_q [R][n_q_heads][head_dim] (bf16, after RoPE)
 * of each sequence's span, against the context's page tables and pool, with
 * span row i of sequence b at position d_base[b] + i attending positions
 * 0..d_base[b]+i. Writes d_out [R][n_q_heads*head_dim] bf16. */
int sdv_op_attention(sdv_ctx *ctx, int layer, const void *d_q, const int32_t *d_row_off, const int32_t *d_base,
                     int B, int max_span, void *d_out, void *stream);

/* Phase timing (cf. [TS] phase counters). While enabled, sdv_spec_forward
 * records CUDA events around each launch group on its stream; this removes
 * the launch overlap between kernels, so durations are those of each kernel
 * run on its own. Groups: 0 prepare/embed, 1 QKV GEMM, 2 attention, 3 O GEMM,
 * 4 gate/up GEMM, 5 down GEMM, 6 LM-head GEMM. */
int sdv_profile_enable(sdv_ctx *ctx, int on);

/* Synchronise, add the elapsed milliseconds and launch counts of every
 * recorded group into h_ms[7] and h_count[7], and clear the record. */
int sdv_profile_read(sdv_ctx *ctx, float *h_ms, int32_t *h_count);

/* Device timeline, for profiling inside a captured or timed step without
 * changing its launches. With d_buf non-null, later sdv_spec_forward calls
 * write %globaltimer stamps (nanoseconds) into it; entries of events that did
 * not happen keep their old value. The buffer is cut into regions of
 * 8192 CTAs x 16 stamps (1,048,576 bytes), one per launch of a forward:
 * layer l uses region 5l for its attention and 5l + 1 + p for its GEMM
 * launches (p = 0 QKV, 1 O, 2 gate/up, 3 down); the LM head uses region
 * 5 n_layers. CTA c of a launch writes d_buf[region * 131072 + c * 16 + e]; a
 * launch with more than 8192 CTAs, or whose region lies past the buffer, is
 * not traced.
 *   GEMM launches: e = 0 CTA start, 1 activations ready (after the wait on
 *   the previous kernel), 2 first stage landed, 3 last MMA issued,
 *   4 accumulator ready, 5 partial parked, 6 all partials of the tile parked,
 *   7 rows finished, 8 CTA end; for the first three passes p of four rows of
 *   the first warp: 9 + 2p the rows' partials summed, 10 + 2p the rows written.
 *   Attention (CTA in launch order): e = 0 start, 1 Q and page ids in, 2 first
 *   chunk landed, 3 chunks done, 4 the CTA states of its cluster in place,
 *   5 cluster merge done, 6 CTA end, 10 second chunk landed, 11 second chunk
 *   computed, 12 last chunk landed; the CTA merging across key groups:
 *   13 merge started, 14 group weights staged, 15 first element summed,
 *   8 merge done.
 * At least 5 regions (1,310,720 bytes), else SDV_ERR_ARG. The buffer
 * (uint64, 8-byte aligned) stays the caller's; d_buf = NULL stops tracing.
 * The pages have no counterpart of this call: it is instrumentation. */
int sdv_fwd_trace(sdv_ctx *ctx, void *d_buf, size_t bytes);

/* Paged attention without any device allocation, for callers that cannot
 * call cudaMalloc: code running while a CUDA graph is being captured,
 * plug-in interfaces that are handed only their input and output buffers,
 * and deployments whose device memory is fixed at start-up. The pages have
 * no counterpart of this call; it is a variant of sdv_op_attention that needs
 * neither a context nor a workspace.
 *   Inputs: d_q [R][n_q_heads][head_dim] bf16 (after RoPE); d_kv_layer, one
 *   layer of a KV pool laid out as in sdv_kv_pool_bytes ([n_pages][2][n_kv_heads]
 *   [page_size][head_dim] bf16); d_page_table [B][pages_per_seq] int32;
 *   d_row_off [B+1] and d_base [B] as in sdv_op_attention. Output: d_out
 *   [R][n_q_heads*head_dim] bf16.
 *   Scratch: a file-scope device array of 8 MiB, held by every GPU that loads
 *   the library until the process exits. The first call on a device resolves
 *   that array's device address and sets kernel attributes; make that first
 *   call before any stream capture. The resolved address is kept for the life
 *   of the process: calls on a device after cudaDeviceReset are not
 *   supported. All calls share the array, so calls that overlap on the GPU
 *   race (calls on different devices do not share it); each call clears the
 *   status word and the group counters it uses.
 *   Limits: B <= 64, head_dim 64 or 128, every L_b + S_b <= max_context <=
 *   pages_per_seq * page_size, and the scratch the shapes need (about
 *   B * ceil(max_context/1024) * n_q_heads * min(max_span,
 *   64*n_kv_heads/n_q_heads) * (4*head_dim + 8) bytes) within 8 MiB; beyond it
 *   the call returns SDV_ERR_CAPACITY and enqueues nothing.
 *   Device-side errors go to a status word in the scratch, read with
 *   sdv_noalloc_status: a sequence whose span is longer than max_span
 *   (SDV_ERR_ARG) or passes max_context (SDV_ERR_CAPACITY) gets NaN rows; a
 *   page id outside [0, n_pages) reads as zero K/V rows and sets
 *   SDV_ERR_CAPACITY. No device memory is allocated or freed. */
int sdv_paged_attention_noalloc(const void *d_q, const void *d_kv_layer, const int32_t *d_page_table,
                                int pages_per_seq, int page_size, int n_pages, const int32_t *d_row_off,
                                const int32_t *d_base, int B, int n_q_heads, int n_kv_heads, int head_dim,
                                int max_span, int max_context, void *d_out, void *stream);

/* Synchronise the current device, copy the status word of the last
 * sdv_paged_attention_noalloc call on it to *h_status (SDV_OK if none ran) and
 * clear it. Allocates nothing. The pages have no counterpart of this call. */
int sdv_noalloc_status(int32_t *h_status);

/* Speculation cost governor ([TS] SpeculationCostGovernor and the paragraphs on
 * the shared governor): a host-side policy, one per (model, drafter, device),
 * that decides before each step whether it drafts, from the measured time of
 * earlier steps; no GPU work. Rules: verdicts compare ms per committed token of
 * speculative steps with the plain baseline (the mean over the last
 * baseline_samples plain samples); a probe is probe_steps speculative steps,
 * after a loss reprobe_steps; a loss parks drafting for first_park tokens,
 * doubling per further loss up to max_park, and a win resets that; a probe
 * ends early, lost, after zero_accept_end speculative steps in a row accepted
 * nothing; while a win holds, the governor parks as soon as the last
 * hold_window speculative steps average a loss, and re-measures the baseline
 * with remeasure_steps plain steps every remeasure_every speculative steps; a
 * speculative step that proposed nothing counts as one token; parked steps
 * feed the baseline except the first; the governor starts with remeasure_steps
 * plain calibration steps. */
typedef struct sdv_governor sdv_governor; /* opaque host state */
typedef struct {
    int probe_steps;      /* 8 */
    int reprobe_steps;    /* 3 */
    int first_park;       /* 32 tokens */
    int max_park;         /* 256 tokens */
    int hold_window;      /* 8 */
    int remeasure_every;  /* 64 */
    int remeasure_steps;  /* 3 */
    int zero_accept_end;  /* 4 */
    int baseline_samples; /* 64 */
} sdv_governor_cfg;
typedef struct {
    float plain_ms_per_tok; /* the baseline, or -1 before any plain sample */
    float spec_ms_per_tok;  /* over every speculative sample, or -1 */
    int wins, losses, parked_steps;
    int state;              /* 0 calibrate, 1 probe, 2 hold, 3 re-measure, 4 parked */
} sdv_governor_report;

/* cfg NULL: the values above. Values < 1, or max_park < first_park: SDV_ERR_ARG. */
int sdv_governor_create(const sdv_governor_cfg *cfg, sdv_governor **out);
int sdv_governor_destroy(sdv_governor *g);
/* *h_speculate = 1 if the next step drafts, 0 for a plain one-row step. */
int sdv_governor_decide(sdv_governor *g, int32_t *h_speculate);
/* The finished step: whether it drafted, its device time, tokens committed
 * (summed over the batch), drafts proposed and accepted. */
int sdv_governor_record(sdv_governor *g, int speculative, float ms, int committed, int drafted, int accepted);
/* A new request: the park left is capped at first_park and the backoff is
 * forgotten; a loss already recorded keeps the next probe short. */
int sdv_governor_new_request(sdv_governor *g);
int sdv_governor_stats(sdv_governor *g, sdv_governor_report *out);

#ifdef __cplusplus
}
#endif
#endif /* SDV_H */
