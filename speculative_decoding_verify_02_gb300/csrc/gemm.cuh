// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05), used for
// every dense projection of the verify forward: Y[rows][out] = X[rows][in] . W[out][in]^T.
//
// The verify span has few rows (K+1 per sequence, <= 128 in all), so the weight
// matrix is the tcgen05 A operand (M = 128 output features per tile, streamed
// from HBM by TMA with 128-byte swizzle) and the activations are the B operand
// (N = rows padded to 16/32/64/128, read from L2), held as a bf16 hi/lo pair:
// the planes are adjacent rows of the B tile, so one MMA of width 2N per k step
// covers both and the epilogue adds the halves. Activations keep about 16
// significant bits while the weights stay exactly bf16. The accumulator sits in
// TMEM. Warp roles: warp 4 issues TMA, warp 5 issues MMAs, warps 0-3 run the
// epilogue from tcgen05.ld. When K is split, the splits of one tile form a
// thread-block cluster: each CTA parks its fp32 partial in its own shared
// memory, and after a cluster barrier CTA q reduces rows q*ceil(R/splits)...
// over distributed shared memory, adding the splits in split order. Every
// output element's reduction order therefore depends only on the weight
// shape, never on how many rows are present.
#pragma once

#include "common.cuh"

namespace sdv {

enum EpiKind : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_LMHEAD = 3 };

struct GemmArgs {
    int kind;
    int tiles, splits, kps, k_blocks;  // output tiles, K splits, k-blocks per split, total k-blocks (64 wide)
    int l2_ahead;                      // k-blocks prefetched into L2 beyond the shared-memory stages
    int deep_ring;                     // host: launched with the deep stage ring
    int n_out;                         // valid output features (ffn for SwiGLU)
    int rows_cap;                      // rows of the activation / ss buffers (plane stride in rows)
    const int *nrows;                  // device: rows present (R)
    int *status;
    // rstd of the RMSNorm feeding this GEMM (QKV, SwiGLU, LM head): from sum-of-squares parts
    const float *ss_in;
    int ss_tiles, hidden;
    float eps;
    // QKV epilogue
    int nq, nkv, D, q_tiles, k_tiles, qk_norm;
    const bf16 *q_gain, *k_gain;
    const float2 *rope;                // [positions][D/2] (cos, sin)
    int rope_rows;
    const int *row_seq, *row_pos, *page_table;
    int pages_per_seq, page_size, n_pages;
    bf16 *q_out, *kv_layer;            // q_out: [2 planes][rows_cap][nq][D]
    // sliding-window layer: ring size, the layer's backup of the slots a span overwrites
    // ([max_batch][max_span][K|V][nkv][D]), the sequences' lengths before the span
    int swa_window, max_span;
    bf16 *swa_backup;
    const int *seq_base;
    // residual epilogue
    float *x;
    bf16 *xb;                          // [2 planes][rows_cap][hidden]
    const bf16 *g_next;
    float *ss_out;
    // SwiGLU epilogue
    bf16 *h_out;                       // [2 planes][rows_cap][ffn]
    // LM-head epilogue
    unsigned long long *keys;
    float *logits;
    int *argmax_out, *done_counter;
    int vocab;
    // sampled verify: per-sequence temperatures ([max_batch], <= 0 = greedy) or nullptr, and the
    // key of the row noise (the rows' sequences and positions come from row_seq / row_pos)
    const float *temperature;
    unsigned long long seed;
    unsigned long long *trace;         // optional timeline: 16 %globaltimer stamps per CTA, or nullptr
};

__device__ __forceinline__ void gemm_stamp(const GemmArgs &a, int ev) {
    if (a.trace) a.trace[static_cast<size_t>(blockIdx.x) * 16 + ev] = globaltimer();
}

// Shared memory given to the stage ring of one GEMM CTA. 104 KB lets two CTAs share an SM (the
// next kernel's CTAs then start streaming weights while this one finishes). A launch whose grid
// fits on the SMs one CTA each may take the deep ring instead (200 KB: twice the weight bytes in
// flight per SM; four stages instead of two at N = 128). The gate/up projection does (its 152
// tiles of the 4B shape fill the SMs exactly): at batch 1 it streams at 8.1 instead of 6.2 TB/s
// between first and last MMA. So does the down projection, with the split count at which all its
// clusters of 200 KB CTAs are resident at once.
#ifndef SDV_GEMM_STAGE_KB
#define SDV_GEMM_STAGE_KB 104
#endif
constexpr int kDeepRingKB = 200;

template <int N, int STAGE_KB = SDV_GEMM_STAGE_KB>
struct GemmShape {
    static constexpr int BM = 128, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_PLANE = N * BK * 2;      // one of the hi / lo planes
    static constexpr int B_BYTES = 2 * B_PLANE;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_RAW = (STAGE_KB * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 16 ? 16 : STAGES_RAW;
    // The hi and lo planes are adjacent in the B stage (N rows each), so one MMA of width 2N
    // covers both: hi product in accumulator columns [0, N), lo product in [N, 2N). One MMA per
    // 16-wide k step instead of two: the tensor core's cost is per instruction at these widths.
    static constexpr int TMEM_COLS = 2 * N < 32 ? 32 : 2 * N;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
    static constexpr uint32_t IDESC = idesc_bf16(128, N);
    static constexpr uint32_t IDESC2 = idesc_bf16(128, 2 * N);
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert(B_PLANE % 1024 == 0, "B planes must keep 1024-byte alignment");
    // one MMA covers both planes: 2N accumulator columns, a legal kind::f16 width for M = 128
    static_assert(2 * N % 16 == 0 && 2 * N <= 256, "MMA width 2N must be a multiple of 16, at most 256");
    static_assert(TMEM_COLS >= 2 * N && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation must hold 2N columns");
    static_assert(2 * TMEM_COLS <= 512, "two co-resident CTAs must fit in the SM's 512 TMEM columns");
    // the fp32 row tile [N][128] that the epilogue parks reuses the stage memory
    static_assert(N * 128 * 4 <= STAGES * STAGE_BYTES, "parked row tile must fit in the stage ring");
    static_assert(STAGE_KB > 112 || 2 * (SMEM_BYTES + 1024) <= 227 * 1024, "two CTAs per SM must fit in shared memory");
    static_assert(SMEM_BYTES + 2048 <= 227 * 1024, "one CTA must fit in shared memory");
};

constexpr int kGemmThreads = 192;
constexpr int kMaxSplits = 8;  // K splits of a tile: one thread-block cluster (portable size)

// ------------------------------------------------------------------ epilogues
// One warp finishes one row at a time. Lane l holds features l, l+32, l+64 and
// l+96 of the 128-feature tile in x[0..3]: every rotate-half pair of a head and
// every gate/up pair of the SwiGLU tile then sits inside one lane, and the row
// reductions (head norm, sum of squares, argmax) are warp reductions. The code
// is small on purpose: each SM runs one CTA of a launch, with a cold
// instruction cache.

struct EpiSmem {
    float rstd[128];
    int last;
};

// Per-layer arguments of the row epilogues (the rest comes from GemmArgs).
struct EpiLayer {
    const bf16 *q_gain, *k_gain;  // QKV: head-norm gains
    bf16 *kv_layer;               // QKV: this layer's KV pool
    const bf16 *g_next;           // residual: gain of the RMSNorm that consumes x
};

// What the QKV epilogue of one row reads besides the accumulator: its position, the RoPE
// (cos, sin) pairs of the lane's features and, for K and V tiles, the page holding the position.
// Loaded while the MMAs run, so the row's finish does not wait on global memory.
struct QkvRow {
    int pos, page, span_row;  // span_row: the row's index in its sequence's span (sliding-window backup)
    float2 c0, c1;
};

__device__ __forceinline__ int qkv_section(const GemmArgs &a, int tile, int &fbase) {
    if (tile < a.q_tiles) {
        fbase = tile * 128;
        return 0;
    }
    if (tile < a.q_tiles + a.k_tiles) {
        fbase = (tile - a.q_tiles) * 128;
        return 1;
    }
    fbase = (tile - a.q_tiles - a.k_tiles) * 128;
    return 2;
}

__device__ __forceinline__ QkvRow qkv_row_load(const GemmArgs &a, int tile, int r, int lane) {
    int fbase;
    const int section = qkv_section(a, tile, fbase);
    QkvRow q;
    q.pos = a.row_pos[r];
    q.page = -1;
    q.c0 = q.c1 = make_float2(1.f, 0.f);
    if (section < 2) {
        const int p = q.pos < 0 ? 0 : (q.pos >= a.rope_rows ? a.rope_rows - 1 : q.pos);
        if (a.D == 128) {
            q.c0 = a.rope[static_cast<size_t>(p) * 64 + lane];
            q.c1 = a.rope[static_cast<size_t>(p) * 64 + lane + 32];
        } else {
            q.c0 = a.rope[static_cast<size_t>(p) * 32 + lane];
        }
    }
    q.span_row = -1;
    if (section > 0) {
        // a sliding-window layer keeps one window of positions in a ring: position p in slot
        // p % window, whose pages are the sequence's first window / page_size page-table entries
        const int seq = a.row_seq[r];
        const int slot_idx = (a.swa_window > 0 ? q.pos % a.swa_window : q.pos) / a.page_size;
        if (seq >= 0 && q.pos >= 0 && slot_idx < a.pages_per_seq)
            q.page = a.page_table[static_cast<size_t>(seq) * a.pages_per_seq + slot_idx];
        if (a.swa_backup != nullptr && seq >= 0) q.span_row = q.pos - a.seq_base[seq];
    }
    return q;
}

// head-norm gains of the lane's features (row-independent): D = 128 features l + 32i; D = 64
// g[0], g[1] = dims l, l + 32 (both heads of the tile share them)
__device__ __forceinline__ void qkv_gains(const GemmArgs &a, const EpiLayer &el, int tile, int lane, float (&g)[4]) {
    int fbase;
    const int section = qkv_section(a, tile, fbase);
    const bf16 *gain = section == 0 ? el.q_gain : el.k_gain;
#pragma unroll
    for (int i = 0; i < 4; ++i) g[i] = 1.f;
    if (section < 2 && a.qk_norm) {
        if (a.D == 128) {
#pragma unroll
            for (int i = 0; i < 4; ++i) g[i] = __bfloat162float(gain[lane + 32 * i]);
        } else {
            g[0] = __bfloat162float(gain[lane]);
            g[1] = __bfloat162float(gain[lane + 32]);
        }
    }
}

__device__ __forceinline__ void epi_qkv_core(const GemmArgs &a, const EpiLayer &el, float rstd, int tile, int r,
                                             int lane, float (&x)[4], const QkvRow &q, const float (&g)[4]) {
    const int D = a.D;
    const int dsh = D == 128 ? 7 : 6;  // head_dim is 64 or 128: head and dim of a feature by shift and mask
    int fbase;  // first feature of the tile inside its section (0 = q, 1 = k, 2 = v)
    const int section = qkv_section(a, tile, fbase);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] *= rstd;
    const int pos = q.pos;
    if (section < 2) {
        if (D == 128) {  // one head: dims l, l+32, l+64, l+96; pairs (l, l+64), (l+32, l+96)
            if (a.qk_norm) {
                const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
                const float sc = rsqrtf(ss / 128.f + a.eps);
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] *= sc * g[i];
            }
            const float2 c0 = q.c0, c1 = q.c1;
            const float y0 = x[0] * c0.x - x[2] * c0.y, y2 = x[2] * c0.x + x[0] * c0.y;
            const float y1 = x[1] * c1.x - x[3] * c1.y, y3 = x[3] * c1.x + x[1] * c1.y;
            x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
        } else {  // D == 64, two heads: (x0, x1) dims l, l+32 of one head, (x2, x3) of the next
            if (a.qk_norm) {
                const float sa = rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1]) / 64.f + a.eps);
                const float sb = rsqrtf(warp_sum(x[2] * x[2] + x[3] * x[3]) / 64.f + a.eps);
                x[0] *= sa * g[0]; x[1] *= sa * g[1]; x[2] *= sb * g[0]; x[3] *= sb * g[1];
            }
            const float2 c = q.c0;
            const float y0 = x[0] * c.x - x[1] * c.y, y1 = x[1] * c.x + x[0] * c.y;
            const float y2 = x[2] * c.x - x[3] * c.y, y3 = x[3] * c.x + x[2] * c.y;
            x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
        }
    }
    if (section == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int fs = fbase + lane + 32 * i;
            const size_t o = (static_cast<size_t>(r) * a.nq + (fs >> dsh)) * D + (fs & (D - 1));
            const Bf16Pair pr = split_bf16(x[i]);
            a.q_out[o] = pr.hi;
            a.q_out[o + static_cast<size_t>(a.rows_cap) * a.nq * D] = pr.lo;
        }
        return;
    }
    const int page = q.page;
    if (page < 0 || page >= a.n_pages) {
        if (lane == 0) set_status(a.status, SDV_ERR_CAPACITY);
        return;
    }
    // sliding-window layer: the slot about to be written holds position pos - window, which other
    // rows of this span may still attend and a rejection must give back; keep it first
    const int slot = (a.page_size & (a.page_size - 1)) == 0 ? pos & (a.page_size - 1) : pos % a.page_size;
    bf16 *keep = nullptr;
    if (a.swa_backup != nullptr && q.span_row >= 0 && q.span_row < a.max_span)
        keep = a.swa_backup + ((static_cast<size_t>(a.row_seq[r]) * a.max_span + q.span_row) * 2 + (section - 1)) *
                                  a.nkv * D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int fs = fbase + lane + 32 * i;
        const size_t off =
            (((static_cast<size_t>(page) * 2 + (section - 1)) * a.nkv + (fs >> dsh)) * a.page_size + slot) * D +
            (fs & (D - 1));
        if (keep != nullptr) keep[fs] = el.kv_layer[off];
        el.kv_layer[off] = __float2bfloat16(x[i]);
    }
}

__device__ __forceinline__ void epi_qkv_row(const GemmArgs &a, const EpiLayer &el, float rstd, int tile, int r,
                                            int lane, float (&x)[4]) {
    float g[4];
    qkv_gains(a, el, tile, lane, g);
    epi_qkv_core(a, el, rstd, tile, r, lane, x, qkv_row_load(a, tile, r, lane), g);
}

// residual-add epilogue of one row: xr = the row's residual values of the lane's features,
// gn = the next RMSNorm's gains of those features (0 past n_out)
__device__ __forceinline__ void epi_resid_core(const GemmArgs &a, int tile, int r, int lane, const float (&x)[4],
                                               const float (&xr)[4], const float (&gn)[4]) {
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int F = tile * 128 + lane + 32 * i;
        if (F < a.n_out) {
            const size_t o = static_cast<size_t>(r) * a.hidden + F;
            const float xn = xr[i] + x[i];
            a.x[o] = xn;
            const Bf16Pair pr = split_bf16(xn * gn[i]);
            a.xb[o] = pr.hi;
            a.xb[o + static_cast<size_t>(a.rows_cap) * a.hidden] = pr.lo;
            sq += xn * xn;
        }
    }
    sq = warp_sum(sq);
    if (lane == 0) a.ss_out[static_cast<size_t>(tile) * a.rows_cap + r] = sq;
}

__device__ __forceinline__ void resid_row_load(const GemmArgs &a, int tile, int r, int lane, float (&xr)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int F = tile * 128 + lane + 32 * i;
        xr[i] = F < a.n_out ? __ldcg(&a.x[static_cast<size_t>(r) * a.hidden + F]) : 0.f;
    }
}

__device__ __forceinline__ void resid_gains(const GemmArgs &a, const EpiLayer &el, int tile, int lane, float (&gn)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int F = tile * 128 + lane + 32 * i;
        gn[i] = F < a.n_out ? __bfloat162float(el.g_next[F]) : 0.f;
    }
}

// xs: the row's 128 residual values already staged in shared memory, or nullptr to read them
__device__ __forceinline__ void epi_resid_row(const GemmArgs &a, const EpiLayer &el, int tile, int r, int lane,
                                              float (&x)[4], const float *xs = nullptr) {
    float xr[4], gn[4];
    if (xs) {
#pragma unroll
        for (int i = 0; i < 4; ++i) xr[i] = xs[lane + 32 * i];
    } else {
        resid_row_load(a, tile, r, lane, xr);
    }
    resid_gains(a, el, tile, lane, gn);
    epi_resid_core(a, tile, r, lane, x, xr, gn);
}

__device__ __forceinline__ void epi_swiglu_row(const GemmArgs &a, float rstd, int tile, int r, int lane,
                                               float (&x)[4]) {
    // gate features tile*64 + (l, l+32) in x0, x1; the matching up features in x2, x3
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int F = tile * 64 + lane + 32 * i;
        if (F < a.n_out) {
            const float gt = x[i] * rstd, up = x[i + 2] * rstd;
            const size_t o = static_cast<size_t>(r) * a.n_out + F;
            const Bf16Pair pr = split_bf16(__fdividef(gt, 1.f + __expf(-gt)) * up);
            a.h_out[o] = pr.hi;
            a.h_out[o + static_cast<size_t>(a.rows_cap) * a.n_out] = pr.lo;
        }
    }
}

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): the output function, and output i of the
// stream keyed k, mix64(k + (i + 1) * golden gamma).
__device__ __forceinline__ unsigned long long splitmix_mix(unsigned long long z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
__device__ __forceinline__ unsigned long long splitmix_at(unsigned long long k, unsigned long long i) {
    return splitmix_mix(k + (i + 1ull) * 0x9E3779B97F4A7C15ull);
}

// Gumbel noise of vocabulary entry v in the stream of one row: u = ((x >> 41) + 1/2) 2^-23 is a
// 23-bit uniform strictly inside (0, 1) that float32 holds exactly; g = -log(-log u).
__device__ __forceinline__ float row_gumbel(unsigned long long row_key, int v) {
    const unsigned long long xr = splitmix_at(row_key, static_cast<unsigned long long>(v));
    const float u = (static_cast<float>(xr >> 41) + 0.5f) * 1.1920928955078125e-07f;
    return -logf(-logf(u));
}

__device__ __forceinline__ void epi_lmhead_row(const GemmArgs &a, float rstd, int tile, int r, int lane,
                                               float (&x)[4]) {
    // sampled rows: the argmax of logit / T + g(seed, sequence, position, v) (Gumbel-max draw)
    float T = 0.f;
    unsigned long long rkey = 0;
    if (a.temperature != nullptr) {
        const int seq = a.row_seq[r];
        T = seq >= 0 ? a.temperature[seq] : 0.f;
        if (T > 0.f) {
            rkey = splitmix_at(splitmix_at(a.seed, static_cast<unsigned long long>(seq)),
                               static_cast<unsigned long long>(a.row_pos[r]));
        }
    }
    uint32_t best = 0, bidx = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // ascending vocabulary index: the first maximum is the lowest index
        const int v = tile * 128 + lane + 32 * i;
        if (v < a.vocab) {
            const float y = x[i] * rstd;
            if (a.logits != nullptr) a.logits[static_cast<size_t>(r) * a.vocab + v] = y;
            const float score = T > 0.f ? y / T + row_gumbel(rkey, v) : y;
            const uint32_t u = orderable(score);
            if (bidx == 0xffffffffu || u > best) {
                best = u;
                bidx = static_cast<uint32_t>(v);
            }
        }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, best);
    const uint32_t idx = __reduce_min_sync(0xffffffffu, best == m ? bidx : 0xffffffffu);
    if (lane == 0 && idx != 0xffffffffu)
        atomicMax(&a.keys[r], (static_cast<unsigned long long>(m) << 32) | (0xffffffffull - idx));
}

template <int KIND>
__device__ __forceinline__ void epi_row(const GemmArgs &a, const EpiLayer &el, const EpiSmem &es, int tile, int r,
                                        int lane, float (&x)[4]) {
    if constexpr (KIND == EPI_QKV) epi_qkv_row(a, el, es.rstd[r], tile, r, lane, x);
    else if constexpr (KIND == EPI_RESID) epi_resid_row(a, el, tile, r, lane, x);
    else if constexpr (KIND == EPI_SWIGLU) epi_swiglu_row(a, es.rstd[r], tile, r, lane, x);
    else epi_lmhead_row(a, es.rstd[r], tile, r, lane, x);
}

// Accumulator rows c0..c0+31 of this warp's 32 output features: hi-plane product (columns
// [0, n)) plus lo-plane product (columns [n, 2n)).
__device__ __forceinline__ void acc_load(uint32_t base, int c0, int n, float (&v)[32]) {
    if (n == 16) {  // one 32-column load holds both halves
        tmem_ld32(base, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] += v[16 + j];
        return;
    }
    float w[32];
    tmem_ld32(base + c0, v);
    tmem_ld32(base + n + c0, w);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += w[j];
}

// ------------------------------------------------------------------ kernel
template <int KIND>
__device__ __forceinline__ void load_a(uint8_t *sa, const CUtensorMap *tmA0, const CUtensorMap *tmA1,
                                       const CUtensorMap *tmA2, uint64_t *bar, const GemmArgs &a, int tile, int kc,
                                       uint64_t pol) {
    if constexpr (KIND == EPI_SWIGLU) {
        // rows 0-63: gate features tile*64.., rows 64-127: the same up features
        tma_load_2d_hint(sa, tmA0, bar, kc, tile * 64, pol);
        tma_load_2d_hint(sa + 8192, tmA1, bar, kc, tile * 64, pol);
    } else if constexpr (KIND == EPI_QKV) {
        if (tile < a.q_tiles)
            tma_load_2d_hint(sa, tmA0, bar, kc, tile * 128, pol);
        else if (tile < a.q_tiles + a.k_tiles)
            tma_load_2d_hint(sa, tmA1, bar, kc, (tile - a.q_tiles) * 128, pol);
        else
            tma_load_2d_hint(sa, tmA2, bar, kc, (tile - a.q_tiles - a.k_tiles) * 128, pol);
    } else {
        tma_load_2d_hint(sa, tmA0, bar, kc, tile * 128, pol);
    }
}

template <int KIND>
__device__ __forceinline__ void prefetch_a(const CUtensorMap *tmA0, const CUtensorMap *tmA1, const CUtensorMap *tmA2,
                                           const GemmArgs &a, int tile, int kc) {
    if constexpr (KIND == EPI_SWIGLU) {
        tma_prefetch_2d(tmA0, kc, tile * 64);
        tma_prefetch_2d(tmA1, kc, tile * 64);
    } else if constexpr (KIND == EPI_QKV) {
        if (tile < a.q_tiles)
            tma_prefetch_2d(tmA0, kc, tile * 128);
        else if (tile < a.q_tiles + a.k_tiles)
            tma_prefetch_2d(tmA1, kc, (tile - a.q_tiles) * 128);
        else
            tma_prefetch_2d(tmA2, kc, (tile - a.q_tiles - a.k_tiles) * 128);
    } else {
        tma_prefetch_2d(tmA0, kc, tile * 128);
    }
}


template <int N, int KIND, int RING_KB = SDV_GEMM_STAGE_KB>
__global__ void __launch_bounds__(kGemmThreads, 2)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    using S = GemmShape<N, RING_KB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full_bar[S::STAGES], empty_bar[S::STAGES], accum_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ EpiSmem es;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / a.splits, split = blockIdx.x % a.splits;
    const int kb0 = split * a.kps;
    const int kb1 = min(kb0 + a.kps, a.k_blocks);
    const int nk = kb1 - kb0;
    const bool clustered = a.splits > 1;

    if (threadIdx.x == 0) {
        gemm_stamp(a, 0);
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&accum_bar, 1);
        fence_mbar_init();
        es.last = 0;
    }
    if (warp == 5) {
        tmem_alloc(&tmem_base_s, S::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&tmA0);
        prefetch_tensormap(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // Let the next kernel in the stream start its prologue now.
    pdl_trigger();

    // the accumulator tile as [N rows][128 features] fp32, in the stage memory (free once the
    // accumulator is final); in a cluster the other CTAs read it over DSMEM.
    float *red = reinterpret_cast<float *>(smem);

    if (warp == 4) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            // Weight tiles do not depend on the previous kernel: start streaming before the wait.
            const int pre = min(nk, S::STAGES);
            for (int i = 0; i < pre; ++i) {
                mbar_arrive_expect_tx(&full_bar[i], S::STAGE_BYTES);
                load_a<KIND>(smem + i * S::STAGE_BYTES, &tmA0, &tmA1, &tmA2, &full_bar[i], a, tile, (kb0 + i) * 64,
                             pol_w);
            }
            // optionally pull further weight tiles into L2 while the previous kernel runs
            const int ahead = min(nk, pre + a.l2_ahead);
            for (int i = pre; i < ahead; ++i) prefetch_a<KIND>(&tmA0, &tmA1, &tmA2, a, tile, (kb0 + i) * 64);
            pdl_wait();  // activations come from the previous kernel
            gemm_stamp(a, 1);
            for (int i = 0; i < pre; ++i)
                tma_load_3d(smem + i * S::STAGE_BYTES + S::A_BYTES, &tmB, &full_bar[i], (kb0 + i) * 64, 0, 0);
            int issued = pre;
            bool timed_out = false;
            for (int i = pre; i < nk; ++i) {
                const int s = i % S::STAGES;
                const uint32_t ph = (i / S::STAGES) & 1;
                if (!mbar_wait(&empty_bar[s], ph ^ 1)) {
                    set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
                    timed_out = true;
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[s], S::STAGE_BYTES);
                uint8_t *sa = smem + s * S::STAGE_BYTES;
                const int kc = (kb0 + i) * 64;
                load_a<KIND>(sa, &tmA0, &tmA1, &tmA2, &full_bar[s], a, tile, kc, pol_w);
                tma_load_3d(sa + S::A_BYTES, &tmB, &full_bar[s], kc, 0, 0);
                issued = i + 1;
            }
            if (timed_out) {
                // error path: the copies already issued must land before this CTA may leave (its
                // shared memory goes to the next CTA); each stage's last issued phase, bounded
                for (int j = max(0, issued - S::STAGES); j < issued; ++j)
                    if (!mbar_wait(&full_bar[j % S::STAGES], (j / S::STAGES) & 1)) break;
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            for (int i = 0; i < nk; ++i) {
                const int s = i % S::STAGES;
                const uint32_t ph = (i / S::STAGES) & 1;
                if (!mbar_wait(&full_bar[s], ph)) {
                    set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
                    break;
                }
                tc_fence_after();
                if (i == 0) gemm_stamp(a, 2);
                const uint64_t ad = sw128_desc(smem_u32(smem + s * S::STAGE_BYTES));
                const uint64_t bd = sw128_desc(smem_u32(smem + s * S::STAGE_BYTES + S::A_BYTES));  // hi rows, then lo
#pragma unroll
                for (int k = 0; k < 4; ++k) umma_bf16(tmem, ad + 2 * k, bd + 2 * k, S::IDESC2, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty_bar[s]);
            }
            gemm_stamp(a, 3);
            umma_commit(&accum_bar);
        }
    }

    // ---------------- epilogue warps 0-3. Rows of the tile this CTA finishes: all R, or its share
    // [s0, s1) of a split tile. Warp w takes rows s0 + w + 4j; the first kPreRows of them get
    // their row data (residual, RoPE, page) loaded while the MMAs still run.
    constexpr int kPreRows = 4;
    int R = 0, s0 = 0, s1 = 0;
    float pre_x[kPreRows][4];  // EPI_RESID: residual values of the lane's features
    QkvRow pre_q[kPreRows];    // EPI_QKV
    float gl[4];               // row-independent gains (QKV head norm, or the next RMSNorm)
    if (warp < 4) {
        pdl_wait();
        R = *a.nrows;
        if (R > N) {
            set_status(a.status, SDV_ERR_ARG);
            R = N;
        }
        if constexpr (KIND != EPI_RESID) {
            const int r = threadIdx.x;
            if (r < N) {
                float s = 0.f;
                if (r < R) {
                    for (int t = 0; t < a.ss_tiles; ++t) s += a.ss_in[static_cast<size_t>(t) * a.rows_cap + r];
                    s = rsqrtf(s / static_cast<float>(a.hidden) + a.eps);
                }
                es.rstd[r] = s;
            }
        }
        s1 = R;
        if (clustered) {
            const int per = (R + a.splits - 1) / a.splits;
            s0 = min(R, static_cast<int>(cluster_ctarank()) * per);
            s1 = min(R, s0 + per);
        }
        const EpiLayer el{a.q_gain, a.k_gain, a.kv_layer, a.g_next};
        if constexpr (KIND == EPI_RESID) {
            resid_gains(a, el, tile, lane, gl);
#pragma unroll
            for (int j = 0; j < kPreRows; ++j) {
                const int r = s0 + warp + 4 * j;
                if (r < s1) resid_row_load(a, tile, r, lane, pre_x[j]);
            }
        } else if constexpr (KIND == EPI_QKV) {
            qkv_gains(a, el, tile, lane, gl);
#pragma unroll
            for (int j = 0; j < kPreRows; ++j) {
                const int r = s0 + warp + 4 * j;
                if (r < s1) pre_q[j] = qkv_row_load(a, tile, r, lane);
            }
        }
        if (!mbar_wait(&accum_bar, 0)) set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
        tc_fence_after();
        if (threadIdx.x == 0) gemm_stamp(a, 4);
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        // park the partial as [row][lane][4]: feature 32 i + l at l * 4 + i, so that the lane that
        // finishes features l, l+32, l+64, l+96 of a row reads them as one 16-byte vector
        const int f = threadIdx.x, fpos = (f & 31) * 4 + (f >> 5);
        float v[32];
        for (int c0 = 0; c0 < R; c0 += 32) {
            acc_load(taddr, c0, N, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < R) red[(c0 + j) * 128 + fpos] = v[j];
        }
    }
    // every partial of the tile is parked in shared memory (of each CTA of the cluster)
    if (threadIdx.x == 0) gemm_stamp(a, 5);
    if (clustered) cluster_sync();
    else if (warp < 4) named_bar_sync(1, 128);
    if (threadIdx.x == 0) gemm_stamp(a, 6);
    if (warp < 4) {
        const EpiLayer el{a.q_gain, a.k_gain, a.kv_layer, a.g_next};
        const uint32_t red_local = smem_u32(red);
        // four rows per pass, their loads issued together
        for (int p = 0; s0 + warp + 16 * p < s1; ++p) {
            float x[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = s0 + warp + 16 * p + 4 * u;
#pragma unroll
                for (int i = 0; i < 4; ++i) x[u][i] = 0.f;
                if (r < s1) {
                    if (clustered) {
                        // every split's 16 bytes in flight together, then summed in split order
                        float4 xs[kMaxSplits];
#pragma unroll
                        for (int q = 0; q < kMaxSplits; ++q)
                            if (q < a.splits)
                                xs[q] = ld_dsmem_f4(mapa_shared(red_local, static_cast<uint32_t>(q)) + r * 512 + lane * 16);
#pragma unroll
                        for (int q = 0; q < kMaxSplits; ++q) {  // fixed split order
                            if (q < a.splits) {
                                x[u][0] += xs[q].x;
                                x[u][1] += xs[q].y;
                                x[u][2] += xs[q].z;
                                x[u][3] += xs[q].w;
                            }
                        }
                    } else {
                        const float4 xv = *reinterpret_cast<const float4 *>(&red[r * 128 + lane * 4]);
                        x[u][0] = xv.x;
                        x[u][1] = xv.y;
                        x[u][2] = xv.z;
                        x[u][3] = xv.w;
                    }
                }
            }
            if (threadIdx.x == 0 && p < 3) gemm_stamp(a, 9 + 2 * p);  // the pass's partials in registers
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = s0 + warp + 16 * p + 4 * u;
                if (r < s1) {
                    if constexpr (KIND == EPI_RESID) {
                        if (p == 0) {
                            epi_resid_core(a, tile, r, lane, x[u], pre_x[u], gl);
                        } else {
                            float xr[4];
                            resid_row_load(a, tile, r, lane, xr);
                            epi_resid_core(a, tile, r, lane, x[u], xr, gl);
                        }
                    } else if constexpr (KIND == EPI_QKV) {
                        epi_qkv_core(a, el, es.rstd[r], tile, r, lane, x[u],
                                     p == 0 ? pre_q[u] : qkv_row_load(a, tile, r, lane), gl);
                    } else {
                        epi_row<KIND>(a, el, es, tile, r, lane, x[u]);
                    }
                }
            }
            if (threadIdx.x == 0 && p < 3) gemm_stamp(a, 10 + 2 * p);  // the pass's rows written
        }
    }
    if (threadIdx.x == 0) gemm_stamp(a, 7);
    // this CTA's reads of the others' partials are done; it leaves only once every CTA of the
    // cluster has arrived (no CTA leaves while its partial may still be read)
    if (clustered) cluster_arrive();
    if constexpr (KIND == EPI_LMHEAD) {
        if (warp < 4) {
            __threadfence();
            named_bar_sync(1, 128);
            if (threadIdx.x == 0)
                es.last = (atomicAdd(a.done_counter, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
            named_bar_sync(1, 128);
            if (es.last) {
                __threadfence();
                const int r = threadIdx.x;
                if (r < R) {
                    const unsigned long long k = atomicAdd(&a.keys[r], 0ull);
                    a.argmax_out[r] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
                }
                if (threadIdx.x == 0) *a.done_counter = 0;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
    if (clustered) cluster_wait();
    if (threadIdx.x == 0) gemm_stamp(a, 8);
}

}  // namespace sdv
