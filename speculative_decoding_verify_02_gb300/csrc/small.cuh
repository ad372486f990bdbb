// Small kernels of the step: forward preparation (embedding gather, row
// bookkeeping, attention work list), greedy acceptance, page reservation and
// LIFO rewind, the n-gram history/hash index, and the span proposer.
#pragma once

#include "common.cuh"

namespace sdv {

// Device-side state held in the workspace.
struct DevState {
    int *status;
    int *seq_len;       // [max_batch] cache length
    int *n_pages;       // [max_batch] pages held
    int *page_table;    // [max_batch][pages_per_seq]
    int *free_stack;    // [n_pages]
    int *free_top;      // [1]
    int *nrows;         // [1] rows of the current forward
    int *seq_base;      // [max_batch] length before the current forward
    int *row_off;       // [max_batch+1] copy of the current forward's offsets
    int *row_seq;       // [rows_cap]
    int *row_pos;       // [rows_cap]
    int4 *work;         // attention work list: (b | group << 16, L_b, S_b, first row of b)
    int *work_off;      // [max_batch+1]
    int *n_work;        // [1]
    // n-gram / loop state
    int *hist;          // [max_batch][ngram_cap]
    int *hist_len;      // [max_batch]
    ulonglong2 *ng_keys;  // [max_batch][ng_orders][ng_slots]: n-token context, order n = 1..ng_orders
    int *ng_vals;         // [max_batch][ng_orders][ng_slots]: position of its most recent follower
    int *cur_tok, *generated, *budget, *kcur;  // [max_batch]
    int *swa_keep;      // [max_batch] rows of the last forward's span kept by the last rewind (sliding window)
    int swa_window;     // > 0: the model has sliding-window layers
    int max_batch, pages_per_seq, page_size, n_pages_total, max_rows, max_span, work_cap;
    int ngram_cap, ng_slots, ng_orders;
};

// An n-gram context of up to six tokens, 21 bits each, packed exactly: tokens 0-2 in x, 3-5 in y.
// x never has its top bit set, so an all-ones x marks an empty slot.
constexpr unsigned long long kEmptyKey = 0xffffffffffffffffull;
constexpr int kNgramMaxOrder = 6;
constexpr int kNgramTokenBits = 21;

__device__ __forceinline__ uint32_t ng_hash(ulonglong2 key, int slots) {
    const unsigned long long h = key.x * 0x9E3779B97F4A7C15ull ^ (key.y + 0x632BE59BD9B4E019ull) * 0xC2B2AE3D27D4EB4Full;
    return static_cast<uint32_t>(h >> 32) & static_cast<uint32_t>(slots - 1);
}

// ------------------------------------------------------------------ init / reset
__global__ void init_state_kernel(DevState s) {
    const int tid = blockIdx.x * blockDim.x + threadIdx.x, nth = gridDim.x * blockDim.x;
    for (int i = tid; i < s.n_pages_total; i += nth) s.free_stack[i] = s.n_pages_total - 1 - i;
    for (int i = tid; i < s.max_batch * s.pages_per_seq; i += nth) s.page_table[i] = -1;
    for (int i = tid; i < s.max_batch; i += nth) {
        s.seq_len[i] = 0;
        s.n_pages[i] = 0;
        s.hist_len[i] = 0;
        s.cur_tok[i] = 0;
        s.generated[i] = 0;
        s.budget[i] = 0;
        s.kcur[i] = 1;
    }
    const long long nslots = static_cast<long long>(s.max_batch) * s.ng_orders * s.ng_slots;
    for (long long i = tid; i < nslots; i += nth) s.ng_keys[i] = make_ulonglong2(kEmptyKey, 0ull);
    if (tid == 0) {
        *s.free_top = s.n_pages_total;
        *s.status = 0;
        *s.nrows = 0;
        *s.n_work = 0;
    }
}

// ------------------------------------------------------------------ forward preparation
struct PrepArgs {
    DevState s;
    const int *tokens;   // [R]
    const int *row_off;  // [B+1] (caller's)
    const int *base;     // [B] explicit cache bases (attention op) or nullptr (forward)
    int B, max_rows, max_span, chunk;
    int embed;           // 1: forward (gather embeddings, advance lengths)
    const bf16 *E;       // [vocab][H]
    const bf16 *g0;      // first RMSNorm gain [H]
    float *x;            // [rows_cap][H]
    bf16 *xb;            // [2 planes: hi, lo][rows_cap][H]
    float *ss;           // [ss_tiles][rows_cap]
    unsigned long long *keys;  // [rows_cap]
    int H, vocab, rows_cap;
};

// Block 0: validate the spans, record bases/offsets/row maps, advance lengths,
// build the attention work list. Blocks 1..max_rows: embed row blockIdx.x-1.
// It does not let its dependents start early: every later kernel of the forward starts after it
// has finished, so what it (and any kernel before it) wrote may be read before their own wait.
__global__ void prepare_kernel(PrepArgs p) {
    pdl_wait();
    DevState &s = p.s;
    __shared__ int ok_s;
    __shared__ int wo_s[257];
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) {
            int ok = p.row_off[0] == 0;
            int R = p.row_off[p.B];
            if (R < 0 || R > p.max_rows) ok = 0;
            int nw = 0;
            for (int b = 0; b < p.B && ok; ++b) {
                const int S = p.row_off[b + 1] - p.row_off[b];
                if (S < 0 || S > p.max_span) {
                    ok = 0;
                    break;
                }
                const int L = p.base ? p.base[b] : s.seq_len[b];
                if (S > 0) {
                    if (L < 0 || static_cast<long long>(L + S) > static_cast<long long>(s.n_pages[b]) * s.page_size) {
                        set_status(s.status, SDV_ERR_CAPACITY);
                        ok = 0;
                        break;
                    }
                }
                wo_s[b] = nw;
                nw += S > 0 ? (L + S + p.chunk - 1) / p.chunk : 0;
            }
            if (ok && nw > s.work_cap) ok = 0;
            if (!ok) {
                set_status(s.status, SDV_ERR_ARG);
                R = 0;
                nw = 0;
                for (int b = 0; b <= p.B; ++b) wo_s[b] = 0;
            }
            wo_s[p.B] = nw;
            ok_s = ok;
            *s.nrows = R;
            *s.n_work = nw;
        }
        __syncthreads();
        const int ok = ok_s;
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
            const int L = p.base ? p.base[b] : s.seq_len[b];
            const int r0 = ok ? p.row_off[b] : 0, r1 = ok ? p.row_off[b + 1] : 0;
            s.seq_base[b] = L;
            s.row_off[b] = r0;
            s.work_off[b] = wo_s[b];
            for (int r = r0; r < r1; ++r) {
                s.row_seq[r] = b;
                s.row_pos[r] = L + (r - r0);
            }
            if (ok && p.embed) s.seq_len[b] = L + (r1 - r0);
        }
        if (threadIdx.x == 0) {
            s.row_off[p.B] = ok ? p.row_off[p.B] : 0;
            s.work_off[p.B] = wo_s[p.B];
        }
        __syncthreads();  // seq_base of every sequence is written
        for (int b = 0; b < p.B; ++b) {
            const int w0 = wo_s[b], n = wo_s[b + 1] - w0;
            if (n == 0) continue;
            const int L = p.base ? p.base[b] : s.seq_base[b];
            const int r0 = p.row_off[b], S = p.row_off[b + 1] - r0;
            for (int c = threadIdx.x; c < n; c += blockDim.x) s.work[w0 + c] = make_int4(b | (c << 16), L, S, r0);
        }
        for (int r = threadIdx.x; r < p.rows_cap; r += blockDim.x) p.keys[r] = 0ull;
        return;
    }
    if (!p.embed) return;
    const int r = blockIdx.x - 1;
    if (r >= p.row_off[p.B] || r >= p.max_rows) return;
    int tok = p.tokens[r];
    if (tok < 0 || tok >= p.vocab) {
        set_status(s.status, SDV_ERR_DEVICE);
        tok = 0;
    }
    // every load first (independent), then the per-128-feature sums of squares
    __shared__ float red[4][64];
    const bf16 *e = p.E + static_cast<size_t>(tok) * p.H;
    const int ntile = (p.H + 127) / 128;
    constexpr int kMaxTiles = 64;  // hidden <= 8192
    float vals[kMaxTiles];
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
        const int f = t * 128 + threadIdx.x;
        vals[t] = (t < ntile && f < p.H) ? __bfloat162float(e[f]) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t) {
        const int f = t * 128 + threadIdx.x;
        if (t < ntile && f < p.H) {
            p.x[static_cast<size_t>(r) * p.H + f] = vals[t];
            const Bf16Pair pr = split_bf16(vals[t] * __bfloat162float(p.g0[f]));
            p.xb[static_cast<size_t>(r) * p.H + f] = pr.hi;
            p.xb[(static_cast<size_t>(p.rows_cap) + r) * p.H + f] = pr.lo;
        }
        if (t < ntile) {
            const float sq = warp_sum(vals[t] * vals[t]);
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5][t] = sq;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < ntile; t += blockDim.x)
        p.ss[static_cast<size_t>(t) * p.rows_cap + r] = (red[0][t] + red[1][t]) + (red[2][t] + red[3][t]);
}

// ------------------------------------------------------------------ accept
struct AcceptArgs {
    DevState s;
    const int *tokens, *row_off, *argmax;
    int B, max_commit, adaptive, k_max;
    int *n_accept, *committed, *n_commit, *new_len;
};

__global__ void accept_kernel(AcceptArgs p) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    DevState &s = p.s;
    const int r0 = p.row_off[b], S = p.row_off[b + 1] - r0;
    if (S <= 0) {
        p.n_accept[b] = -1;
        p.n_commit[b] = 0;
        p.new_len[b] = -1;
        return;
    }
    const int k = S - 1;
    int m = 0;
    while (m < k && p.tokens[r0 + 1 + m] == p.argmax[r0 + m]) ++m;
    if (m + 1 > p.max_commit) set_status(s.status, SDV_ERR_ARG);
    for (int i = 0; i <= m && i < p.max_commit; ++i) p.committed[b * p.max_commit + i] = p.argmax[r0 + i];
    p.n_accept[b] = m;
    p.n_commit[b] = m + 1;
    p.new_len[b] = s.seq_len[b] - S + m + 1;
    // loop state: next current token, tokens generated, adaptive draft length
    s.cur_tok[b] = p.argmax[r0 + m];
    s.generated[b] += m + 1;
    if (p.adaptive && k > 0) s.kcur[b] = (m == k) ? min(s.kcur[b] + 2, p.k_max) : max(s.kcur[b] - 1, 1);
}

// ------------------------------------------------------------------ pages
__global__ void ensure_kernel(DevState s, const int *required, int B) {
    pdl_trigger();
    pdl_wait();
    __shared__ int need_s[256], off_s[256], ok_s, top_s;
    if (threadIdx.x == 0) {
        int ok = 1, total = 0;
        const int top = *s.free_top;
        for (int b = 0; b < B; ++b) {
            const int req = required[b];
            int need = 0;
            if (req >= 0) {
                const int pages = (req + s.page_size - 1) / s.page_size;
                if (pages > s.pages_per_seq) ok = 0;
                need = max(0, pages - s.n_pages[b]);
            }
            need_s[b] = need;
            off_s[b] = total;
            total += need;
        }
        if (total > top) ok = 0;
        if (!ok) set_status(s.status, SDV_ERR_CAPACITY);
        ok_s = ok;
        top_s = top;
        if (ok) *s.free_top = top - total;
    }
    __syncthreads();
    if (!ok_s) return;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int n0 = s.n_pages[b];
        for (int j = 0; j < need_s[b]; ++j)
            s.page_table[b * s.pages_per_seq + n0 + j] = s.free_stack[top_s - 1 - (off_s[b] + j)];
        s.n_pages[b] = n0 + need_s[b];
    }
}

__global__ void rewind_kernel(DevState s, const int *length, int B) {
    pdl_trigger();
    pdl_wait();
    __shared__ int rel_s[256], off_s[256], ok_s, top_s;
    if (threadIdx.x == 0) {
        int ok = 1;
        for (int b = 0; b < B; ++b) {
            const int len = length[b];
            rel_s[b] = 0;
            if (len < 0) continue;
            if (len > s.seq_len[b]) {
                ok = 0;
                continue;
            }
            // sliding-window rings keep only what the last forward evicted
            if (s.swa_window > 0 && len < s.seq_base[b] && s.seq_len[b] > s.swa_window) {
                ok = 0;
                continue;
            }
            const int keep = (len + s.page_size - 1) / s.page_size;
            rel_s[b] = max(0, s.n_pages[b] - keep);
        }
        int total = 0;
        for (int b = B - 1; b >= 0; --b) {
            off_s[b] = total;
            total += rel_s[b];
        }
        if (!ok) set_status(s.status, SDV_ERR_ARG);
        ok_s = ok;
        top_s = *s.free_top;
        if (ok) *s.free_top = top_s + total;
    }
    __syncthreads();
    if (!ok_s) return;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const int len = length[b];
        if (len < 0) continue;
        const int n = s.n_pages[b];
        for (int j = 0; j < rel_s[b]; ++j) {
            const int slot = n - 1 - j;
            s.free_stack[top_s + off_s[b] + j] = s.page_table[b * s.pages_per_seq + slot];
            s.page_table[b * s.pages_per_seq + slot] = -1;
        }
        s.n_pages[b] = n - rel_s[b];
        s.seq_len[b] = len;
    }
    // rows of the last forward kept (the rest are restored in the sliding-window rings)
    if (s.swa_window > 0)
        for (int b = threadIdx.x; b < B; b += blockDim.x) {
            const int len = length[b];
            s.swa_keep[b] = len < 0 ? 1 << 30 : len - s.seq_base[b];
        }
}

// [TS] sliding-window caches and rollback: for every local layer and sequence, the slots of the
// last forward's rejected rows (span rows at or past the kept count) get back the positions they
// held, from the layer's backup; a full acceptance restores nothing. Grid (B, n_layers).
__global__ void swa_restore_kernel(DevState s, bf16 *pool, size_t layer_stride, const unsigned long long local_mask,
                                   const bf16 *backup, size_t backup_layer_stride, int nkv, int D, int B) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, l = blockIdx.y;
    if (b >= B || !((local_mask >> l) & 1ull)) return;
    const int li = __popcll(local_mask & ((1ull << l) - 1ull));  // index among the local layers
    const int p = s.seq_base[b], S = s.row_off[b + 1] - s.row_off[b], keep = max(0, s.swa_keep[b]);
    const int W = s.swa_window, P = s.page_size;
    const int row = D * nkv;  // elements of one K (or V) row of all heads
    for (int j = keep; j < S && j < s.max_span; ++j) {
        const int u = p + j - W;  // the position span row j evicted
        if (u < 0) continue;
        const int page = s.page_table[static_cast<size_t>(b) * s.pages_per_seq + ((p + j) % W) / P];
        if (page < 0 || page >= s.n_pages_total) continue;
        const bf16 *src = backup + li * backup_layer_stride + (static_cast<size_t>(b) * s.max_span + j) * 2 * row;
        bf16 *dst = pool + l * layer_stride;
        for (int e = threadIdx.x; e < 2 * row; e += blockDim.x) {
            const int kv = e / row, h = (e % row) / D, d = e % D;
            dst[(((static_cast<size_t>(page) * 2 + kv) * nkv + h) * P + (p + j) % P) * D + d] = src[e];
        }
    }
}

__global__ void reset_seq_kernel(DevState s, int b) {
    pdl_wait();
    if (threadIdx.x == 0) {
        const int top = *s.free_top, n = s.n_pages[b];
        for (int j = 0; j < n; ++j) {
            const int slot = n - 1 - j;
            s.free_stack[top + j] = s.page_table[b * s.pages_per_seq + slot];
            s.page_table[b * s.pages_per_seq + slot] = -1;
        }
        *s.free_top = top + n;
        s.n_pages[b] = 0;
        s.seq_len[b] = 0;
        s.hist_len[b] = 0;
        s.cur_tok[b] = 0;
        s.generated[b] = 0;
        s.budget[b] = 0;
        s.kcur[b] = 1;
    }
    for (int i = threadIdx.x; i < s.ng_orders * s.ng_slots; i += blockDim.x)
        s.ng_keys[static_cast<size_t>(b) * s.ng_orders * s.ng_slots + i] = make_ulonglong2(kEmptyKey, 0ull);
}

// ------------------------------------------------------------------ n-gram index and proposer
__device__ __forceinline__ size_t ng_table(const DevState &s, int b, int n) {
    return (static_cast<size_t>(b) * s.ng_orders + (n - 1)) * s.ng_slots;
}

__device__ __forceinline__ bool ng_insert(DevState &s, int b, int n, ulonglong2 key, int val) {
    ulonglong2 *keys = s.ng_keys + ng_table(s, b, n);
    int *vals = s.ng_vals + ng_table(s, b, n);
    uint32_t h = ng_hash(key, s.ng_slots);
    for (int probe = 0; probe < s.ng_slots; ++probe) {
        const ulonglong2 k = keys[h];
        if (k.x == kEmptyKey || (k.x == key.x && k.y == key.y)) {
            keys[h] = key;
            vals[h] = val;
            return true;
        }
        h = (h + 1) & static_cast<uint32_t>(s.ng_slots - 1);
    }
    return false;
}

__device__ __forceinline__ int ng_lookup(const DevState &s, int b, int n, ulonglong2 key) {
    const ulonglong2 *keys = s.ng_keys + ng_table(s, b, n);
    const int *vals = s.ng_vals + ng_table(s, b, n);
    uint32_t h = ng_hash(key, s.ng_slots);
    for (int probe = 0; probe < s.ng_slots; ++probe) {
        const ulonglong2 k = keys[h];
        if (k.x == key.x && k.y == key.y) return vals[h];
        if (k.x == kEmptyKey) return -1;
        h = (h + 1) & static_cast<uint32_t>(s.ng_slots - 1);
    }
    return -1;
}

// The context h[end - n .. end - 1] as a packed key.
__device__ __forceinline__ ulonglong2 ng_key(const int *h, int end, int n) {
    unsigned long long w[2] = {0ull, 0ull};
    for (int i = 0; i < n; ++i)
        w[i / 3] |= static_cast<unsigned long long>(static_cast<uint32_t>(h[end - n + i])) << (kNgramTokenBits * (i % 3));
    return make_ulonglong2(w[0], w[1]);
}

// Append tokens to sequence b's history; each new token at position L completes the contexts
// h[L-n .. L-1] (n = 1 .. orders), which now map to L, their most recent follower.
__global__ void ngram_commit_kernel(DevState s, const int *tokens, const int *counts, int B, int stride) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B || s.ngram_cap <= 0) return;
    int *h = s.hist + static_cast<size_t>(b) * s.ngram_cap;
    int L = s.hist_len[b];
    const int n = counts[b];
    for (int i = 0; i < n; ++i) {
        if (L >= s.ngram_cap) {
            set_status(s.status, SDV_ERR_CAPACITY);
            break;
        }
        const int tok = tokens[static_cast<size_t>(b) * stride + i];
        if (tok < 0 || tok >= (1 << kNgramTokenBits)) {
            set_status(s.status, SDV_ERR_DEVICE);
            break;
        }
        for (int o = 1; o <= s.ng_orders && o <= L; ++o)
            if (!ng_insert(s, b, o, ng_key(h, L, o), L)) set_status(s.status, SDV_ERR_CAPACITY);
        h[L] = tok;
        ++L;
    }
    s.hist_len[b] = L;
}

__global__ void gen_init_kernel(DevState s, const int *first, const int *budget, int B, int k_init) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    s.cur_tok[b] = first[b];
    s.generated[b] = 1;
    s.budget[b] = budget[b];
    s.kcur[b] = k_init;
}

// One block; thread b builds sequence b's span, thread 0 packs the offsets.
// n-gram drafter: the longest order n in [ng_req, ng_orders] whose last-n-token context occurred
// earlier with a follower; its most recent occurrence gives up to k drafts.
__global__ void propose_kernel(DevState s, int drafter, const int *table, int table_stride, int B, int max_span,
                               int ng_req, int *tokens, int *row_off, int *required) {
    pdl_trigger();
    pdl_wait();
    __shared__ int len_s[257], off_s[257];
    const int b = threadIdx.x;
    int n = 0, src = -1;  // drafts: n tokens from hist[src..] (n-gram) or table[...]
    bool active = false;
    if (b < B) {
        const int g = s.generated[b];
        active = g < s.budget[b];
        if (active) {
            int k = min(s.kcur[b], s.budget[b] - g - 1);
            k = min(k, max_span - 1);
            if (drafter == SDV_DRAFT_NGRAM && k > 0 && s.ngram_cap > 0) {
                const int L = s.hist_len[b];
                const int *h = s.hist + static_cast<size_t>(b) * s.ngram_cap;
                for (int o = s.ng_orders; o >= ng_req && o >= 1; --o) {
                    if (L < o + 1) continue;
                    const int j = ng_lookup(s, b, o, ng_key(h, L, o));
                    if (j >= o && j < L) {
                        src = j;
                        n = min(k, L - j);
                        break;
                    }
                }
            } else if (drafter == SDV_DRAFT_TABLE && k > 0) {
                src = g;
                n = k;
            }
        }
        len_s[b] = active ? 1 + n : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int i = 0; i < B; ++i) {
            off_s[i] = acc;
            acc += len_s[i];
        }
        off_s[B] = acc;
    }
    __syncthreads();
    for (int i = threadIdx.x; i <= B; i += blockDim.x) row_off[i] = off_s[i];
    if (b < B) {
        required[b] = active ? s.seq_len[b] + 1 + n : -1;
        if (active) {
            const int o = off_s[b];
            tokens[o] = s.cur_tok[b];
            for (int i = 0; i < n; ++i)
                tokens[o + 1 + i] = drafter == SDV_DRAFT_NGRAM
                                        ? s.hist[static_cast<size_t>(b) * s.ngram_cap + src + i]
                                        : table[static_cast<size_t>(b) * table_stride + src + i];
        }
    }
}

}  // namespace sdv
