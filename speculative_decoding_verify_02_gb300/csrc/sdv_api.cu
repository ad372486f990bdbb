// C ABI of the verify path: context creation (workspace carve-out, TMA
// descriptors, RoPE table, empty page pool) and the launch sequences of
// spec_forward, accept, ensure_capacity, rewind, n-gram and propose.
#include <cmath>
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "attention.cuh"
#include "attention_group.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "small.cuh"

using namespace sdv;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct GemmPlan {
    int tiles = 0, k_blocks = 0, splits = 1, kps = 0;
    bool deep = false;  // launched with the deep stage ring (one CTA per SM)
};

constexpr int kRowsCap = 128;     // activation rows held in the workspace (max_rows <= 128)
constexpr int kNs[4] = {16, 32, 64, 128};

int n_index(int max_rows) {
    if (max_rows <= 16) return 0;
    if (max_rows <= 32) return 1;
    if (max_rows <= 64) return 2;
    return 3;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }
int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

GemmPlan make_plan(int tiles, int k_blocks, int sm_count, int fixed_splits = 0) {
    GemmPlan p;
    p.tiles = tiles;
    p.k_blocks = k_blocks;
    // Split K so that tiles x splits covers the SMs; depends only on the weight shape. The
    // splits of a tile run as one thread-block cluster, so at most 8 (the portable size).
    int splits = fixed_splits > 0 ? fixed_splits : ceil_div(sm_count, tiles);
    splits = std::max(1, std::min({splits, std::max(1, k_blocks / 2), 8}));
    p.kps = ceil_div(k_blocks, splits);
    p.splits = ceil_div(k_blocks, p.kps);
    return p;
}

// The down projection's plan: the deep stage ring at one CTA per SM (twice the weight bytes in flight
// of the 104 KB ring: at batch 16 its launch went from 23.8 to 18.9 us a layer, at batch 1 from 13.0
// to 12.0) with the largest split count whose whole grid runs at once: tiles x splits within the SMs
// and every cluster of that many 200 KB CTAs resident together (the clusters need whole free SMs of
// one GPC, so a split count the GPCs cannot hold would run the grid in two waves). The count depends
// only on the weight shape and the device, as batch invariance requires. Without a device to ask,
// the ordinary plan (its buffers are the larger).
GemmPlan deep_plan(int tiles, int k_blocks, int sm_count) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        auto kern = gemm_kernel<16, EPI_RESID, kDeepRingKB>;
        const int smem = GemmShape<16, kDeepRingKB>::SMEM_BYTES;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
            for (int s = kMaxSplits; s >= 2; --s) {
                GemmPlan p = make_plan(tiles, k_blocks, sm_count, s);
                if (p.splits != s || static_cast<long long>(tiles) * s > sm_count) continue;
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(tiles * s);
                cfg.blockDim = dim3(kGemmThreads);
                cfg.dynamicSmemBytes = smem;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = s;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters >= tiles) {
                    p.deep = true;
                    return p;
                }
            }
        }
    }
    cudaGetLastError();
    return make_plan(tiles, k_blocks, sm_count);
}

}  // namespace

struct sdv_ctx {
    sdv_model_cfg m{};
    sdv_cache_cfg c{};
    int device = 0, sm_count = 0;
    sdv_weights w{};
    std::vector<sdv_layer_weights> layers;
    bf16 *pool = nullptr;
    uint8_t *ws = nullptr;
    DevState st{};
    float *x = nullptr, *ss = nullptr;
    bf16 *xb = nullptr, *q = nullptr, *attn_o = nullptr, *h = nullptr;
    int *done_lm = nullptr;
    unsigned long long *keys = nullptr;
    float2 *rope = nullptr;
    std::vector<float2> rope_host;
    float *attn_po = nullptr;
    float2 *attn_pml = nullptr;
    int *attn_cnt = nullptr;
    int attn_splits = 1;
    int attn_group = kAttnGroup;  // key positions per attention group (1024, or 2048 for long sequences)
    int attn_lo = 1;  // attention products with hi/lo pairs (queries and probabilities)
    unsigned long long *trace = nullptr;  // caller's timeline buffer (sdv_fwd_trace), or nullptr
    size_t trace_words = 0;
    int ss_tiles = 0, grp = 0, qrows = 0, work_cap = 0, pages_per_seq = 0, ng_slots = 0;
    size_t layer_stride = 0;  // pool elements per layer
    GemmPlan plan[5];         // qkv, o, gate/up, down, lm head
    std::vector<CUtensorMap> tm_wq, tm_wk, tm_wv, tm_wo, tm_wg, tm_wu, tm_wd;
    CUtensorMap tm_lm{};
    KvMaps tm_kv{};          // the KV pool, one map per kv head (encode_pool)
    bool attn_tma = false;   // attention_group.cuh usable (page size a power of two in [8, 128])
    CUtensorMap tm_xb[4]{}, tm_ao[4]{}, tm_h[4]{};
    bool use_pdl = true;
    int gen_adaptive = 0, gen_kmax = 1;  // adaptive-K settings from sdv_gen_init
    bf16 *swa_backup = nullptr;          // sliding-window layers' evicted-slot backups
    size_t swa_layer_elems = 0;
    unsigned long long swa_mask = 0;     // bit l: layer l is a sliding-window layer
    int ng_min = 2;                      // n-gram lookup: shortest match length and its pmin scaling
    float ng_pmin = 0.f;
    // phase timing
    bool profiling = false;
    std::vector<cudaEvent_t> ev_pool;
    std::vector<std::pair<int, std::pair<int, int>>> ev_marks;  // (group, (start event, stop event))
    size_t ev_used = 0;
    ~sdv_ctx() {
        for (cudaEvent_t e : ev_pool) cudaEventDestroy(e);
    }
};

namespace {
cudaEvent_t next_event(sdv_ctx *ctx) {
    if (ctx->ev_used == ctx->ev_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        ctx->ev_pool.push_back(e);
    }
    return ctx->ev_pool[ctx->ev_used++];
}
// Marks one launch group when profiling; no-op otherwise.
struct PhaseMark {
    sdv_ctx *ctx;
    int group, i0 = -1;
    cudaStream_t st;
    PhaseMark(sdv_ctx *c, int g, cudaStream_t s) : ctx(c), group(g), st(s) {
        if (ctx->profiling) {
            cudaEvent_t e = next_event(ctx);
            if (e) {
                i0 = static_cast<int>(ctx->ev_used - 1);
                cudaEventRecord(e, st);
            }
        }
    }
    ~PhaseMark() {
        if (ctx->profiling && i0 >= 0) {
            cudaEvent_t e = next_event(ctx);
            if (e) {
                cudaEventRecord(e, st);
                ctx->ev_marks.push_back({group, {i0, static_cast<int>(ctx->ev_used - 1)}});
            }
        }
    }
};
}  // namespace

namespace {

enum { P_QKV = 0, P_O = 1, P_GU = 2, P_DOWN = 3, P_LM = 4 };
// Timeline buffer (sdv_fwd_trace): one region of kTraceRegionCtas x 16 stamps per launch of a
// step. Layer l uses regions 5l (attention) and 5l + 1 + p (GEMM of plan p, p < 4); the LM head
// uses region 5 n_layers.
constexpr int kTraceRegionCtas = 8192;
constexpr size_t kTraceRegionWords = static_cast<size_t>(kTraceRegionCtas) * 16;

// Sliding-window layers as a bit mask over layers (bit l set: layer l is local).
unsigned long long local_mask(const sdv_model_cfg &m) {
    unsigned long long mask = 0;
    if (m.swa_window <= 0) return 0;
    for (int l = 0; l < m.n_layers && l < 64; ++l)
        if (m.swa_global_every <= 0 || (l + 1) % m.swa_global_every != 0) mask |= 1ull << l;
    return mask;
}

// n-gram orders indexed per sequence: 1 .. ngram_max_order (0 selects 2).
int ngram_orders(const sdv_cache_cfg &c) { return c.ngram_max_order > 0 ? c.ngram_max_order : 2; }

// Required n-gram match length ([TS] --spec-pmin scales it for the n-gram drafter): linear from
// min_order (pmin 0) to the highest indexed order (pmin 1), rounded half up.
int ngram_required(int min_order, int max_order, float pmin) {
    return min_order + static_cast<int>(std::floor(static_cast<double>(pmin) * (max_order - min_order) + 0.5));
}

// Carve the workspace. With ctx == nullptr only the size is computed.
size_t carve(const sdv_model_cfg &m, const sdv_cache_cfg &c, sdv_ctx *ctx, uint8_t *base, int sm_count) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> uint8_t * {
        off = align_up(off, 256);
        uint8_t *p = base ? base + off : nullptr;
        off += bytes;
        return p;
    };
    const int B = c.max_batch, H = m.hidden, D = m.head_dim, F = m.ffn;
    const int qdim = m.n_q_heads * D, kvdim = m.n_kv_heads * D;
    const int pps = ceil_div(c.max_context, c.page_size);
    const int grp = m.n_q_heads / m.n_kv_heads;
    const int qrows = kAttnRows / grp;
    // attention: CTAs (one cluster) per (key group, kv head), fixed by the configuration (a row's
    // arithmetic must not depend on the span): the largest power of two <= 8 that keeps the grid
    // within four CTAs per SM for a full batch at full context and groups x splits <= 64. Groups
    // hold 1024 positions; where that leaves one CTA per group and doubling the group brings a
    // full-size grid into one wave of CTAs (long single sequences), 2048 (the TMA-fed kernel only).
    int group = kAttnGroup;
    int max_groups = ceil_div(c.max_context, group);
    int splits = 8;
    while (splits > 1 && (static_cast<long long>(B) * max_groups * m.n_kv_heads * splits > 4LL * sm_count ||
                          max_groups * splits > 64))
        splits >>= 1;
    const bool tma_attn = c.page_size >= 8 && c.page_size <= kAttnChunk && (c.page_size & (c.page_size - 1)) == 0 &&
                          m.n_kv_heads <= kMaxKvHeads;
    if (tma_attn && splits == 1 &&
        static_cast<long long>(B) * ceil_div(c.max_context, 2 * kAttnGroup) * m.n_kv_heads <= sm_count) {
        group = 2 * kAttnGroup;
        max_groups = ceil_div(c.max_context, group);
    }
    const int work_cap = ceil_div(static_cast<long long>(c.n_pages) * c.page_size, group) + B;
    const int ng_slots = c.ngram_capacity > 0 ? next_pow2(std::max(16, 2 * c.ngram_capacity)) : 0;
    const int ng_orders = ngram_orders(c);
    const int ss_tiles = ceil_div(H, 128);

    GemmPlan plans[5] = {make_plan((qdim + 2 * kvdim) / 128, ceil_div(H, 64), sm_count),
                         make_plan(ceil_div(H, 128), ceil_div(qdim, 64), sm_count),
                         make_plan(ceil_div(F, 64), ceil_div(H, 64), sm_count),
                         deep_plan(ceil_div(H, 128), ceil_div(F, 64), sm_count),
                         make_plan(ceil_div(m.vocab, 128), ceil_div(H, 64), sm_count)};

    DevState s{};
    s.status = reinterpret_cast<int *>(take(sizeof(int)));
    s.seq_len = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.n_pages = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.page_table = reinterpret_cast<int *>(take(sizeof(int) * static_cast<size_t>(B) * pps));
    s.free_stack = reinterpret_cast<int *>(take(sizeof(int) * static_cast<size_t>(c.n_pages)));
    s.free_top = reinterpret_cast<int *>(take(sizeof(int)));
    s.nrows = reinterpret_cast<int *>(take(sizeof(int)));
    s.seq_base = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.row_off = reinterpret_cast<int *>(take(sizeof(int) * (B + 1)));
    s.row_seq = reinterpret_cast<int *>(take(sizeof(int) * kRowsCap));
    s.row_pos = reinterpret_cast<int *>(take(sizeof(int) * kRowsCap));
    s.work = reinterpret_cast<int4 *>(take(sizeof(int4) * static_cast<size_t>(work_cap)));
    s.work_off = reinterpret_cast<int *>(take(sizeof(int) * (B + 1)));
    s.n_work = reinterpret_cast<int *>(take(sizeof(int)));
    s.hist = reinterpret_cast<int *>(take(sizeof(int) * static_cast<size_t>(B) * std::max(0, c.ngram_capacity)));
    s.hist_len = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.ng_keys = reinterpret_cast<ulonglong2 *>(take(sizeof(ulonglong2) * static_cast<size_t>(B) * ng_orders * ng_slots));
    s.ng_vals = reinterpret_cast<int *>(take(sizeof(int) * static_cast<size_t>(B) * ng_orders * ng_slots));
    s.cur_tok = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.generated = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.budget = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.kcur = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.swa_keep = reinterpret_cast<int *>(take(sizeof(int) * B));
    s.swa_window = m.swa_window > 0 ? m.swa_window : 0;
    s.max_batch = B;
    s.pages_per_seq = pps;
    s.page_size = c.page_size;
    s.n_pages_total = c.n_pages;
    s.max_rows = c.max_rows;
    s.max_span = c.max_span;
    s.work_cap = work_cap;
    s.ngram_cap = c.ngram_capacity;
    s.ng_slots = ng_slots;
    s.ng_orders = ng_orders;

    float *x = reinterpret_cast<float *>(take(sizeof(float) * kRowsCap * H));
    bf16 *xb = reinterpret_cast<bf16 *>(take(sizeof(bf16) * 2 * kRowsCap * H));        // hi, lo planes
    float *ss = reinterpret_cast<float *>(take(sizeof(float) * ss_tiles * kRowsCap));
    bf16 *q = reinterpret_cast<bf16 *>(take(sizeof(bf16) * 2 * kRowsCap * qdim));
    bf16 *ao = reinterpret_cast<bf16 *>(take(sizeof(bf16) * 2 * kRowsCap * qdim));
    bf16 *hb = reinterpret_cast<bf16 *>(take(sizeof(bf16) * 2 * kRowsCap * F));
    // sliding-window backups: per local layer [max_batch][max_span][K|V][nkv][D]
    const int n_local = __builtin_popcountll(local_mask(m));
    const size_t swa_layer = static_cast<size_t>(B) * c.max_span * 2 * kvdim;
    bf16 *swa_backup = reinterpret_cast<bf16 *>(take(sizeof(bf16) * swa_layer * n_local));
    int *done_lm = reinterpret_cast<int *>(take(sizeof(int)));
    auto *keys = reinterpret_cast<unsigned long long *>(take(sizeof(unsigned long long) * kRowsCap));
    float2 *rope = reinterpret_cast<float2 *>(take(sizeof(float2) * static_cast<size_t>(c.max_context) * (D / 2)));
    const size_t nslots = static_cast<size_t>(work_cap) * splits * m.n_kv_heads * grp * qrows;
    float *apo = reinterpret_cast<float *>(take(sizeof(float) * nslots * D));
    float2 *apml = reinterpret_cast<float2 *>(take(sizeof(float2) * nslots));
    int *acnt = reinterpret_cast<int *>(take(sizeof(int) * static_cast<size_t>(B) * m.n_kv_heads * kAttnCluster));

    if (ctx) {
        ctx->st = s;
        ctx->x = x;
        ctx->xb = xb;
        ctx->ss = ss;
        ctx->q = q;
        ctx->attn_o = ao;
        ctx->h = hb;
        for (int i = 0; i < 5; ++i) ctx->plan[i] = plans[i];
        ctx->done_lm = done_lm;
        ctx->swa_backup = swa_backup;
        ctx->swa_layer_elems = swa_layer;
        ctx->swa_mask = local_mask(m);
        ctx->keys = keys;
        ctx->rope = rope;
        ctx->attn_po = apo;
        ctx->attn_pml = apml;
        ctx->attn_cnt = acnt;
        ctx->attn_splits = splits;
        ctx->attn_group = group;
        ctx->ss_tiles = ss_tiles;
        ctx->grp = grp;
        ctx->qrows = qrows;
        ctx->work_cap = work_cap;
        ctx->pages_per_seq = pps;
        ctx->ng_slots = ng_slots;
    }
    return align_up(off, 256);
}

int check_cfg(const sdv_model_cfg *m, const sdv_cache_cfg *c) {
    if (!m || !c) return SDV_ERR_ARG;
    if (m->n_layers <= 0 || m->hidden <= 0 || m->n_q_heads <= 0 || m->n_kv_heads <= 0 || m->ffn <= 0 ||
        m->vocab <= 0)
        return SDV_ERR_ARG;
    if (m->n_q_heads % m->n_kv_heads) return SDV_ERR_ARG;
    if (m->head_dim != 64 && m->head_dim != 128) return SDV_ERR_UNSUPPORTED;
    const int grp = m->n_q_heads / m->n_kv_heads;
    if (grp > 8 || 128 % grp) return SDV_ERR_UNSUPPORTED;
    if ((m->n_q_heads * m->head_dim) % 128 || (m->n_kv_heads * m->head_dim) % 128) return SDV_ERR_UNSUPPORTED;
    if (m->hidden % 8 || m->ffn % 8 || m->hidden > 8192 || m->vocab >= (1 << 30)) return SDV_ERR_UNSUPPORTED;
    if (c->page_size <= 0 || c->n_pages <= 0 || c->max_batch <= 0 || c->max_batch > 256) return SDV_ERR_ARG;
    if (c->max_rows <= 0 || c->max_rows > kRowsCap || c->max_span <= 0 || c->max_span > c->max_rows)
        return SDV_ERR_ARG;
    if (c->max_context <= 0 || c->ngram_capacity < 0) return SDV_ERR_ARG;
    if (c->ngram_max_order < 0 || c->ngram_max_order > kNgramMaxOrder) return SDV_ERR_ARG;
    if (m->swa_window < 0 || m->swa_global_every < 0) return SDV_ERR_ARG;
    if (m->swa_window > 0) {  // a ring of whole pages, never shorter than a span
        if (m->swa_window % c->page_size || m->swa_window < c->max_span) return SDV_ERR_ARG;
        if (m->n_layers > 64) return SDV_ERR_UNSUPPORTED;
    }
    // n-gram contexts pack 21 bits per token
    if (c->ngram_capacity > 0 && m->vocab > (1 << kNgramTokenBits)) return SDV_ERR_UNSUPPORTED;
    return SDV_OK;
}

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 3-D bf16 map over the hi/lo planes of an activation buffer [2][rows][cols]; box = 64 columns x
// box_rows rows x both planes, 128-byte swizzle (the planes land one after the other in shared memory).
bool encode_planes(CUtensorMap *tm, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {cols, rows, 2};
    cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    cuuint32_t box[3] = {64, box_rows, 2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The paged KV pool as a 5-D bf16 tensor [layer * n_pages][K|V][kv_head][slot][dim]; box = 64 dims x
// page_size slots of one (page, K|V, head), 128-byte swizzle.
// One map per kv head over the pool [layer x page][K|V][kv head][slot][dim], dimensions
// [64 dims][slot][64-dim half][K|V][layer x page]: one box = a page's K and V rows of that head,
// both halves, landing as [K|V][half][slot] lines of 128 bytes, so that eight consecutive keys of
// one half sit on eight consecutive swizzle lines (8 KB per box at page size 16, head dim 128).
bool encode_pool(KvMaps *tm, const void *pool, const sdv_model_cfg &m, const sdv_cache_cfg &c) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    const uint64_t D = m.head_dim, P = c.page_size, H = m.n_kv_heads;
    if (H > kMaxKvHeads) return false;
    cuuint64_t dims[5] = {64, P, D / 64, 2, static_cast<cuuint64_t>(m.n_layers) * c.n_pages};
    cuuint64_t strides[4] = {D * 2, 128, H * P * D * 2, 2 * H * P * D * 2};
    cuuint32_t box[5] = {64, static_cast<cuuint32_t>(P), static_cast<cuuint32_t>(D / 64), 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    for (uint64_t h = 0; h < H; ++h) {
        const char *base = static_cast<const char *>(pool) + h * P * D * 2;
        if (enc(&tm->m[h], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<char *>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// 2-D bf16 map over a row-major [rows][cols] matrix; box = 64 columns x box_rows rows, 128-byte swizzle.
bool encode_2d(CUtensorMap *tm, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename... KArgs, typename... Args>
cudaError_t launch(const sdv_ctx *ctx, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ctx->use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(const sdv_ctx *ctx, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t st, int cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (ctx->use_pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int N, int KIND>
cudaError_t launch_gemm_nk(const sdv_ctx *ctx, const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &a2,
                           const CUtensorMap &b, const GemmArgs &args, int grid, cudaStream_t st) {
    // the gate/up projection takes the deep ring when its grid fits on the SMs, one CTA each
    const bool deep = (KIND == EPI_SWIGLU && grid <= ctx->sm_count) || (KIND == EPI_RESID && args.deep_ring);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = deep ? GemmShape<N, kDeepRingKB>::SMEM_BYTES : GemmShape<N>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (ctx->use_pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (args.splits > 1) {  // the K splits of a tile form one cluster
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = args.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    if constexpr (KIND == EPI_SWIGLU || KIND == EPI_RESID)
        if (deep) return cudaLaunchKernelEx(&cfg, gemm_kernel<N, KIND, kDeepRingKB>, a0, a1, a2, b, args);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<N, KIND>, a0, a1, a2, b, args);
}

template <int KIND>
cudaError_t launch_gemm_k(const sdv_ctx *ctx, int nidx, const CUtensorMap &a0, const CUtensorMap &a1,
                          const CUtensorMap &a2, const CUtensorMap &b, const GemmArgs &args, int grid,
                          cudaStream_t st) {
    switch (nidx) {
        case 0: return launch_gemm_nk<16, KIND>(ctx, a0, a1, a2, b, args, grid, st);
        case 1: return launch_gemm_nk<32, KIND>(ctx, a0, a1, a2, b, args, grid, st);
        case 2: return launch_gemm_nk<64, KIND>(ctx, a0, a1, a2, b, args, grid, st);
        default: return launch_gemm_nk<128, KIND>(ctx, a0, a1, a2, b, args, grid, st);
    }
}

cudaError_t launch_gemm(const sdv_ctx *ctx, int nidx, const CUtensorMap &a0, const CUtensorMap &a1,
                        const CUtensorMap &a2, const CUtensorMap &b, const GemmArgs &args, int grid, cudaStream_t st) {
    switch (args.kind) {
        case EPI_QKV: return launch_gemm_k<EPI_QKV>(ctx, nidx, a0, a1, a2, b, args, grid, st);
        case EPI_RESID: return launch_gemm_k<EPI_RESID>(ctx, nidx, a0, a1, a2, b, args, grid, st);
        case EPI_SWIGLU: return launch_gemm_k<EPI_SWIGLU>(ctx, nidx, a0, a1, a2, b, args, grid, st);
        default: return launch_gemm_k<EPI_LMHEAD>(ctx, nidx, a0, a1, a2, b, args, grid, st);
    }
}

// Dynamic shared memory for a kernel, and the largest shared-memory carveout so that two
// CTAs fit on an SM (the default carveout leaves room for one).
template <typename K>
cudaError_t set_smem(K kern, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    return e;
}

template <int N>
cudaError_t set_gemm_smem() {
    cudaError_t e = set_smem(gemm_kernel<N, EPI_QKV>, GemmShape<N>::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(gemm_kernel<N, EPI_RESID>, GemmShape<N>::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(gemm_kernel<N, EPI_SWIGLU>, GemmShape<N>::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(gemm_kernel<N, EPI_LMHEAD>, GemmShape<N>::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(gemm_kernel<N, EPI_SWIGLU, kDeepRingKB>, GemmShape<N, kDeepRingKB>::SMEM_BYTES);
    if (e == cudaSuccess) e = set_smem(gemm_kernel<N, EPI_RESID, kDeepRingKB>, GemmShape<N, kDeepRingKB>::SMEM_BYTES);
    return e;
}

int rc(cudaError_t e) { return e == cudaSuccess ? SDV_OK : SDV_ERR_CUDA; }

// Stamps of launch `region` of the step, or nullptr when tracing is off or the launch has too many CTAs.
unsigned long long *trace_region(const sdv_ctx *ctx, int region, size_t ctas) {
    if (!ctx->trace || ctas > kTraceRegionCtas || ctx->trace_words < kTraceRegionWords * (region + 1)) return nullptr;
    return ctx->trace + kTraceRegionWords * region;
}

GemmArgs base_args(const sdv_ctx *ctx, int kind, int pidx, int layer) {
    GemmArgs a{};
    const GemmPlan &p = ctx->plan[pidx];
    a.kind = kind;
    a.tiles = p.tiles;
    a.splits = p.splits;
    a.kps = p.kps;
    a.k_blocks = p.k_blocks;
    a.deep_ring = p.deep ? 1 : 0;
    a.rows_cap = kRowsCap;
    a.nrows = ctx->st.nrows;
    a.status = ctx->st.status;
    a.ss_in = ctx->ss;
    a.ss_tiles = ctx->ss_tiles;
    a.hidden = ctx->m.hidden;
    a.eps = ctx->m.rms_eps;
    a.trace = trace_region(ctx, pidx == P_LM ? 5 * ctx->m.n_layers : 5 * layer + 1 + pidx,
                           static_cast<size_t>(p.tiles) * p.splits);
    return a;
}

// The backup of local layer l (its index among the local layers).
bf16 *swa_backup_of(const sdv_ctx *ctx, int l) {
    const int li = __builtin_popcountll(ctx->swa_mask & ((1ull << l) - 1ull));
    return ctx->swa_backup + ctx->swa_layer_elems * li;
}

// Paged attention of `layer` over the rows prepared in the device state.
int run_attention(sdv_ctx *ctx, int layer, const bf16 *q, size_t q_plane, bf16 *out, size_t out_plane, int B,
                  int max_span, cudaStream_t st) {
    const sdv_model_cfg &m = ctx->m;
    AttnArgs a{};
    a.q = q;
    a.q_plane = q_plane;
    a.out_plane = out_plane;
    a.kv_layer = ctx->pool + ctx->layer_stride * layer;
    a.page_table = ctx->st.page_table;
    a.pages_per_seq = ctx->pages_per_seq;
    a.page_size = ctx->c.page_size;
    a.n_pages = ctx->c.n_pages;
    a.work = ctx->st.work;
    a.n_work = ctx->st.n_work;
    a.nq = m.n_q_heads;
    a.nkv = m.n_kv_heads;
    a.D = m.head_dim;
    a.grp = ctx->grp;
    a.qrows = ctx->qrows;
    a.scale_log2 = 1.4426950408889634f / std::sqrt(static_cast<float>(m.head_dim));
    a.part_o = ctx->attn_po;
    a.part_ml = ctx->attn_pml;
    a.counters = ctx->attn_cnt;
    a.out = out;
    a.status = ctx->st.status;
    a.splits = ctx->attn_splits;
    a.group = ctx->attn_group;
    a.layer = layer;
    if ((ctx->swa_mask >> layer) & 1ull) {
        a.window = m.swa_window;
        a.max_span = ctx->c.max_span;
        a.swa_backup = swa_backup_of(ctx, layer);
    }
    // the timeline buffer of sdv_fwd_trace, when set (the TMA-fed kernel writes it)
    a.trace = trace_region(ctx, 5 * layer, static_cast<size_t>(ctx->work_cap) * ctx->attn_splits * m.n_kv_heads);
    a.p_lo = ctx->attn_lo;
    if (!ctx->attn_lo) a.q_plane = 0;  // queries as bf16 only
    if (!ctx->attn_tma) {  // 8-CTA clusters per 1024-position group (attention.cuh)
        const dim3 grid(ctx->work_cap * kAttnCluster, m.n_kv_heads);
        a.splits = 1;
        for (int q0 = 0; q0 < max_span; q0 += ctx->qrows) {
            a.q0 = q0;
            cudaError_t e;
            if (m.head_dim == 128)
                e = launch_cluster(ctx, attn_kernel<128>, grid, dim3(kAttnThreads), AttnShape<128>::SMEM, st,
                                   kAttnCluster, a);
            else
                e = launch_cluster(ctx, attn_kernel<64>, grid, dim3(kAttnThreads), AttnShape<64>::SMEM, st,
                                   kAttnCluster, a);
            if (e != cudaSuccess) return SDV_ERR_CUDA;
        }
        return SDV_OK;
    }
    // a cluster of `splits` CTAs per (1024-position group, kv head), chunks pipelined inside each,
    // at most kGrpRows query rows per launch (attention_group.cuh)
    const dim3 grid(ctx->attn_splits, m.n_kv_heads, ctx->work_cap);
    a.qrows = std::max(1, kGrpRows / ctx->grp);
    // Merge across key groups: inside the attention kernel when a group's cluster has at least four
    // CTAs to share the rows (up to kInKernelMergeGroups groups), else by attn_merge_kernel, which
    // is launched only when the configuration allows such sequences.
    a.merge_groups = ctx->attn_splits >= 4 ? kInKernelMergeGroups : 1;
    const bool merge = ceil_div(static_cast<long long>(ctx->c.max_context), ctx->attn_group) > a.merge_groups;
    const dim3 mgrid(ceil_div(kGrpRows, kMergeRows), m.n_kv_heads, B);
    for (int q0 = 0; q0 < max_span; q0 += a.qrows) {
        a.q0 = q0;
        cudaError_t e;
        if (m.head_dim == 128)
            e = launch_cluster(ctx, attn_group_kernel<128>, grid, dim3(kGrpThreads), GrpShape<128>::SMEM, st,
                               ctx->attn_splits, a, ctx->tm_kv);
        else
            e = launch_cluster(ctx, attn_group_kernel<64>, grid, dim3(kGrpThreads), GrpShape<64>::SMEM, st,
                               ctx->attn_splits, a, ctx->tm_kv);
        if (e == cudaSuccess && merge) {
            const int *work_off = ctx->st.work_off;
            if (m.head_dim == 128)
                e = launch(ctx, attn_merge_kernel<128>, mgrid, dim3(kMergeRows * 128 / 4), 0, st, a, work_off);
            else
                e = launch(ctx, attn_merge_kernel<64>, mgrid, dim3(kMergeRows * 64 / 4), 0, st, a, work_off);
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
    }
    return SDV_OK;
}

int prepare(sdv_ctx *ctx, const int32_t *tokens, const int32_t *row_off, const int32_t *base, int B, int max_rows,
            int max_span, int embed, cudaStream_t st) {
    PrepArgs p{};
    p.s = ctx->st;
    p.tokens = tokens;
    p.row_off = row_off;
    p.base = base;
    p.B = B;
    p.max_rows = max_rows;
    p.max_span = max_span;
    p.chunk = ctx->attn_group;
    p.embed = embed;
    p.E = static_cast<const bf16 *>(ctx->w.embed);
    p.g0 = static_cast<const bf16 *>(ctx->layers[0].attn_norm);
    p.x = ctx->x;
    p.xb = ctx->xb;
    p.ss = ctx->ss;
    p.keys = ctx->keys;
    p.H = ctx->m.hidden;
    p.vocab = ctx->m.vocab;
    p.rows_cap = kRowsCap;
    return rc(launch(ctx, prepare_kernel, dim3(embed ? 1 + max_rows : 1), dim3(128), 0, st, p));
}

// Arguments of the QKV projection of layer l (q/k head norm, RoPE, paged K/V write).
GemmArgs qkv_args(const sdv_ctx *ctx, int l) {
    const sdv_model_cfg &m = ctx->m;
    GemmArgs a = base_args(ctx, EPI_QKV, P_QKV, l);
    a.n_out = (m.n_q_heads + 2 * m.n_kv_heads) * m.head_dim;
    a.nq = m.n_q_heads;
    a.nkv = m.n_kv_heads;
    a.D = m.head_dim;
    a.q_tiles = m.n_q_heads * m.head_dim / 128;
    a.k_tiles = m.n_kv_heads * m.head_dim / 128;
    a.qk_norm = m.qk_norm;
    a.rope = ctx->rope;
    a.rope_rows = ctx->c.max_context;
    a.row_seq = ctx->st.row_seq;
    a.row_pos = ctx->st.row_pos;
    a.page_table = ctx->st.page_table;
    a.pages_per_seq = ctx->pages_per_seq;
    a.page_size = ctx->c.page_size;
    a.n_pages = ctx->c.n_pages;
    a.q_out = ctx->q;
    a.q_gain = static_cast<const bf16 *>(ctx->layers[l].q_norm);
    a.k_gain = static_cast<const bf16 *>(ctx->layers[l].k_norm);
    a.kv_layer = ctx->pool + ctx->layer_stride * l;
    if ((ctx->swa_mask >> l) & 1ull) {  // sliding-window layer: ring slots, keep what a span evicts
        a.swa_window = m.swa_window;
        a.max_span = ctx->c.max_span;
        a.swa_backup = swa_backup_of(ctx, l);
        a.seq_base = ctx->st.seq_base;
    }
    return a;
}

}  // namespace

extern "C" {

int sdv_workspace_bytes(const sdv_model_cfg *m, const sdv_cache_cfg *c, size_t *bytes) {
    int r = check_cfg(m, c);
    if (r) return r;
    if (!bytes) return SDV_ERR_ARG;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    *bytes = carve(*m, *c, nullptr, nullptr, sms);
    return SDV_OK;
}

int sdv_kv_pool_bytes(const sdv_model_cfg *m, const sdv_cache_cfg *c, size_t *bytes) {
    int r = check_cfg(m, c);
    if (r) return r;
    if (!bytes) return SDV_ERR_ARG;
    *bytes = static_cast<size_t>(m->n_layers) * c->n_pages * 2 * m->n_kv_heads * c->page_size * m->head_dim * 2;
    return SDV_OK;
}

int sdv_create(const sdv_model_cfg *m, const sdv_cache_cfg *c, const sdv_weights *w, void *d_kv_pool,
               void *d_workspace, void *stream, sdv_ctx **out) {
    int r = check_cfg(m, c);
    if (r) return r;
    if (!w || !w->layers || !w->embed || !w->lm_head || !w->final_norm || !d_kv_pool || !d_workspace || !out)
        return SDV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(d_workspace) % 256 || reinterpret_cast<uintptr_t>(d_kv_pool) % 16)
        return SDV_ERR_ARG;
    for (int l = 0; l < m->n_layers; ++l) {
        const sdv_layer_weights &L = w->layers[l];
        const void *ps[] = {L.attn_norm, L.wq, L.wk, L.wv, L.q_norm, L.k_norm, L.wo, L.ffn_norm, L.w_gate, L.w_up, L.w_down};
        for (const void *p : ps)
            if (!p || reinterpret_cast<uintptr_t>(p) % 16) return SDV_ERR_ARG;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SDV_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, gemm_kernel<16, EPI_QKV>) != cudaSuccess) {
        cudaGetLastError();
        return SDV_ERR_UNSUPPORTED;  // no sm_103a image for this device
    }
    if (!get_encoder()) return SDV_ERR_CUDA;

    sdv_ctx *ctx = new (std::nothrow) sdv_ctx();
    if (!ctx) return SDV_ERR_ARG;
    ctx->m = *m;
    ctx->c = *c;
    ctx->device = dev;
    ctx->sm_count = sms;
    ctx->w = *w;
    ctx->layers.assign(w->layers, w->layers + m->n_layers);
    ctx->w.layers = ctx->layers.data();
    ctx->pool = static_cast<bf16 *>(d_kv_pool);
    ctx->ws = static_cast<uint8_t *>(d_workspace);
    ctx->layer_stride = static_cast<size_t>(c->n_pages) * 2 * m->n_kv_heads * c->page_size * m->head_dim;
    carve(*m, *c, ctx, ctx->ws, sms);

    bool ok = true;
    const int H = m->hidden, D = m->head_dim, F = m->ffn;
    const int qdim = m->n_q_heads * D, kvdim = m->n_kv_heads * D;
    ctx->tm_wq.resize(m->n_layers);
    ctx->tm_wk.resize(m->n_layers);
    ctx->tm_wv.resize(m->n_layers);
    ctx->tm_wo.resize(m->n_layers);
    ctx->tm_wg.resize(m->n_layers);
    ctx->tm_wu.resize(m->n_layers);
    ctx->tm_wd.resize(m->n_layers);
    for (int l = 0; l < m->n_layers && ok; ++l) {
        const sdv_layer_weights &L = ctx->layers[l];
        ok &= encode_2d(&ctx->tm_wq[l], L.wq, qdim, H, 128);
        ok &= encode_2d(&ctx->tm_wk[l], L.wk, kvdim, H, 128);
        ok &= encode_2d(&ctx->tm_wv[l], L.wv, kvdim, H, 128);
        ok &= encode_2d(&ctx->tm_wo[l], L.wo, H, qdim, 128);
        ok &= encode_2d(&ctx->tm_wg[l], L.w_gate, F, H, 64);
        ok &= encode_2d(&ctx->tm_wu[l], L.w_up, F, H, 64);
        ok &= encode_2d(&ctx->tm_wd[l], L.w_down, H, F, 128);
    }
    ok &= encode_2d(&ctx->tm_lm, w->lm_head, m->vocab, H, 128);
    ctx->attn_tma = c->page_size >= 8 && c->page_size <= kAttnChunk && (c->page_size & (c->page_size - 1)) == 0 &&
                    m->n_kv_heads <= kMaxKvHeads;
    if (ctx->attn_tma) ok &= encode_pool(&ctx->tm_kv, d_kv_pool, *m, *c);
    if (m->swa_window > 0 && !ctx->attn_tma) {  // sliding-window layers run on the TMA-fed attention only
        delete ctx;
        return SDV_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < 4 && ok; ++i) {
        ok &= encode_planes(&ctx->tm_xb[i], ctx->xb, kRowsCap, H, kNs[i]);
        ok &= encode_planes(&ctx->tm_ao[i], ctx->attn_o, kRowsCap, qdim, kNs[i]);
        ok &= encode_planes(&ctx->tm_h[i], ctx->h, kRowsCap, F, kNs[i]);
    }
    if (!ok) {
        delete ctx;
        return SDV_ERR_CUDA;
    }

    cudaError_t e = cudaSuccess;
    e = set_gemm_smem<16>();
    if (e == cudaSuccess) e = set_gemm_smem<32>();
    if (e == cudaSuccess) e = set_gemm_smem<64>();
    if (e == cudaSuccess) e = set_gemm_smem<128>();
    if (e == cudaSuccess) e = set_smem(attn_kernel<128>, AttnShape<128>::SMEM);
    if (e == cudaSuccess) e = set_smem(attn_kernel<64>, AttnShape<64>::SMEM);
    if (e == cudaSuccess) e = set_smem(attn_group_kernel<128>, GrpShape<128>::SMEM);
    if (e == cudaSuccess) e = set_smem(attn_group_kernel<64>, GrpShape<64>::SMEM);
    if (e != cudaSuccess) {
        delete ctx;
        return SDV_ERR_CUDA;
    }

    // RoPE table: cos/sin of pos * theta^(-2j/D), in double on the host.
    const int half = D / 2;
    ctx->rope_host.resize(static_cast<size_t>(c->max_context) * half);
    for (int p = 0; p < c->max_context; ++p)
        for (int j = 0; j < half; ++j) {
            const double ang = static_cast<double>(p) * std::pow(static_cast<double>(m->rope_theta), -2.0 * j / D);
            ctx->rope_host[static_cast<size_t>(p) * half + j] =
                make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
        }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t ws_bytes = carve(*m, *c, nullptr, nullptr, sms);
    e = cudaMemsetAsync(ctx->ws, 0, ws_bytes, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ctx->rope, ctx->rope_host.data(), ctx->rope_host.size() * sizeof(float2),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) {
        init_state_kernel<<<64, 256, 0, st>>>(ctx->st);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        delete ctx;
        return SDV_ERR_CUDA;
    }
    *out = ctx;
    return SDV_OK;
}

int sdv_destroy(sdv_ctx *ctx) {
    delete ctx;
    return SDV_OK;
}

int sdv_ensure_capacity(sdv_ctx *ctx, const int32_t *d_required, int B, void *stream) {
    if (!ctx || !d_required || B <= 0 || B > ctx->c.max_batch) return SDV_ERR_ARG;
    return rc(launch(ctx, ensure_kernel, dim3(1), dim3(256), 0, static_cast<cudaStream_t>(stream), ctx->st,
                     d_required, B));
}

}  // extern "C"

namespace {
// The verify forward; temperature == nullptr: per-row argmax, else per-row draws (sampled verify).
int spec_forward_impl(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, int B, int max_rows,
                      int max_span, int32_t *d_argmax, float *d_logits, const float *d_temperature,
                      unsigned long long seed, void *stream) {
    if (!ctx || !d_tokens || !d_row_off || !d_argmax) return SDV_ERR_ARG;
    if (B <= 0 || B > ctx->c.max_batch || max_rows <= 0 || max_rows > ctx->c.max_rows || max_span <= 0 ||
        max_span > ctx->c.max_span || max_span > max_rows)
        return SDV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const sdv_model_cfg &m = ctx->m;
    const int ni = n_index(max_rows);
    int r;
    {
        PhaseMark pm(ctx, 0, st);
        r = prepare(ctx, d_tokens, d_row_off, nullptr, B, max_rows, max_span, 1, st);
    }
    if (r) return r;
    for (int l = 0; l < m.n_layers; ++l) {
        const sdv_layer_weights &L = ctx->layers[l];
        // QKV projection + q/k head norm + RoPE + paged K/V write
        GemmArgs a = qkv_args(ctx, l);
        cudaError_t e;
        {
            PhaseMark pm(ctx, 1, st);
            e = launch_gemm(ctx, ni, ctx->tm_wq[l], ctx->tm_wk[l], ctx->tm_wv[l], ctx->tm_xb[ni], a,
                            ctx->plan[P_QKV].tiles * ctx->plan[P_QKV].splits, st);
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
        {
            PhaseMark pm(ctx, 2, st);
            const size_t plane = static_cast<size_t>(kRowsCap) * m.n_q_heads * m.head_dim;
            r = run_attention(ctx, l, ctx->q, plane, ctx->attn_o, plane, B, max_span, st);
        }
        if (r) return r;
        // O projection + residual; emits bf16(x * g_ffn) and sum-of-squares parts. Its weights
        // (21 MB) are pulled into L2 during the attention, when HBM is otherwise idle.
        a = base_args(ctx, EPI_RESID, P_O, l);
        a.l2_ahead = 64;
        a.n_out = m.hidden;
        a.x = ctx->x;
        a.xb = ctx->xb;
        a.g_next = static_cast<const bf16 *>(L.ffn_norm);
        a.ss_out = ctx->ss;
        {
            PhaseMark pm(ctx, 3, st);
            e = launch_gemm(ctx, ni, ctx->tm_wo[l], ctx->tm_wo[l], ctx->tm_wo[l], ctx->tm_ao[ni], a,
                            ctx->plan[P_O].tiles * ctx->plan[P_O].splits, st);
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
        // gate/up projection + SwiGLU
        a = base_args(ctx, EPI_SWIGLU, P_GU, l);
        a.n_out = m.ffn;
        a.h_out = ctx->h;
        {
            PhaseMark pm(ctx, 4, st);
            e = launch_gemm(ctx, ni, ctx->tm_wg[l], ctx->tm_wu[l], ctx->tm_wg[l], ctx->tm_xb[ni], a,
                            ctx->plan[P_GU].tiles * ctx->plan[P_GU].splits, st);
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
        // down projection + residual; emits bf16(x * g_next) for the next layer (or the final norm)
        a = base_args(ctx, EPI_RESID, P_DOWN, l);
        a.n_out = m.hidden;
        a.x = ctx->x;
        a.xb = ctx->xb;
        a.g_next = static_cast<const bf16 *>(l + 1 < m.n_layers ? ctx->layers[l + 1].attn_norm : ctx->w.final_norm);
        a.ss_out = ctx->ss;
        {
            PhaseMark pm(ctx, 5, st);
            e = launch_gemm(ctx, ni, ctx->tm_wd[l], ctx->tm_wd[l], ctx->tm_wd[l], ctx->tm_h[ni], a,
                            ctx->plan[P_DOWN].tiles * ctx->plan[P_DOWN].splits, st);
        }
        if (e != cudaSuccess) return SDV_ERR_CUDA;
    }
    // final norm (folded as a per-row scale) + LM head + per-row argmax
    GemmArgs a = base_args(ctx, EPI_LMHEAD, P_LM, 0);
    a.keys = ctx->keys;
    a.logits = d_logits;
    a.argmax_out = d_argmax;
    a.done_counter = ctx->done_lm;
    a.vocab = m.vocab;
    a.temperature = d_temperature;
    a.seed = seed;
    a.row_seq = ctx->st.row_seq;
    a.row_pos = ctx->st.row_pos;
    cudaError_t e;
    {
        PhaseMark pm(ctx, 6, st);
        e = launch_gemm(ctx, ni, ctx->tm_lm, ctx->tm_lm, ctx->tm_lm, ctx->tm_xb[ni], a,
                        ctx->plan[P_LM].tiles * ctx->plan[P_LM].splits, st);
    }
    return e == cudaSuccess ? SDV_OK : SDV_ERR_CUDA;
}
}  // namespace

extern "C" {

int sdv_spec_forward(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, int B, int max_rows,
                     int max_span, int32_t *d_argmax, float *d_logits, void *stream) {
    return spec_forward_impl(ctx, d_tokens, d_row_off, B, max_rows, max_span, d_argmax, d_logits, nullptr, 0,
                             stream);
}

int sdv_spec_forward_sampled(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, int B, int max_rows,
                             int max_span, const float *d_temperature, uint64_t seed, int32_t *d_drawn,
                             float *d_logits, void *stream) {
    if (!d_temperature) return SDV_ERR_ARG;
    return spec_forward_impl(ctx, d_tokens, d_row_off, B, max_rows, max_span, d_drawn, d_logits, d_temperature,
                             seed, stream);
}

int sdv_accept_greedy(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_row_off, const int32_t *d_argmax,
                      int B, int max_commit, int32_t *d_n_accept, int32_t *d_committed, int32_t *d_n_commit,
                      int32_t *d_new_len, void *stream) {
    if (!ctx || !d_tokens || !d_row_off || !d_argmax || !d_n_accept || !d_committed || !d_n_commit || !d_new_len)
        return SDV_ERR_ARG;
    if (B <= 0 || B > ctx->c.max_batch || max_commit <= 0) return SDV_ERR_ARG;
    AcceptArgs p{};
    p.s = ctx->st;
    p.tokens = d_tokens;
    p.row_off = d_row_off;
    p.argmax = d_argmax;
    p.B = B;
    p.max_commit = max_commit;
    p.adaptive = ctx->gen_adaptive;
    p.k_max = ctx->gen_kmax;
    p.n_accept = d_n_accept;
    p.committed = d_committed;
    p.n_commit = d_n_commit;
    p.new_len = d_new_len;
    return rc(launch(ctx, accept_kernel, dim3(ceil_div(B, 128)), dim3(128), 0, static_cast<cudaStream_t>(stream), p));
}

int sdv_rewind_cache(sdv_ctx *ctx, const int32_t *d_length, int B, void *stream) {
    if (!ctx || !d_length || B <= 0 || B > ctx->c.max_batch) return SDV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch(ctx, rewind_kernel, dim3(1), dim3(256), 0, st, ctx->st, d_length, B);
    if (e == cudaSuccess && ctx->swa_mask)
        e = launch(ctx, swa_restore_kernel, dim3(B, ctx->m.n_layers), dim3(256), 0, st, ctx->st, ctx->pool,
                   ctx->layer_stride, ctx->swa_mask, static_cast<const bf16 *>(ctx->swa_backup), ctx->swa_layer_elems,
                   ctx->m.n_kv_heads, ctx->m.head_dim, B);
    return rc(e);
}

int sdv_cache_seq_len(sdv_ctx *ctx, int32_t *d_len, void *stream) {
    if (!ctx || !d_len) return SDV_ERR_ARG;
    return rc(cudaMemcpyAsync(d_len, ctx->st.seq_len, sizeof(int) * ctx->c.max_batch, cudaMemcpyDeviceToDevice,
                              static_cast<cudaStream_t>(stream)));
}

int sdv_page_table(sdv_ctx *ctx, int32_t *d_table, int32_t *d_n_pages, int32_t *d_free_top, void *stream) {
    if (!ctx) return SDV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (d_table)
        e = cudaMemcpyAsync(d_table, ctx->st.page_table, sizeof(int) * ctx->c.max_batch * ctx->pages_per_seq,
                            cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && d_n_pages)
        e = cudaMemcpyAsync(d_n_pages, ctx->st.n_pages, sizeof(int) * ctx->c.max_batch, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && d_free_top)
        e = cudaMemcpyAsync(d_free_top, ctx->st.free_top, sizeof(int), cudaMemcpyDeviceToDevice, st);
    return rc(e);
}

int sdv_ngram_commit(sdv_ctx *ctx, const int32_t *d_tokens, const int32_t *d_counts, int B, int stride,
                     void *stream) {
    if (!ctx || !d_tokens || !d_counts || B <= 0 || B > ctx->c.max_batch || stride <= 0) return SDV_ERR_ARG;
    if (ctx->c.ngram_capacity <= 0) return SDV_ERR_UNSUPPORTED;
    return rc(launch(ctx, ngram_commit_kernel, dim3(ceil_div(B, 128)), dim3(128), 0,
                     static_cast<cudaStream_t>(stream), ctx->st, d_tokens, d_counts, B, stride));
}

int sdv_gen_init(sdv_ctx *ctx, const int32_t *d_first, const int32_t *d_budget, int B, int k_init, int adaptive,
                 int k_max, void *stream) {
    if (!ctx || !d_first || !d_budget || B <= 0 || B > ctx->c.max_batch || k_init < 0) return SDV_ERR_ARG;
    if (adaptive && (k_max < 1 || k_init < 1 || k_init > k_max)) return SDV_ERR_ARG;
    ctx->gen_adaptive = adaptive ? 1 : 0;
    ctx->gen_kmax = adaptive ? k_max : std::max(k_init, 1);
    return rc(launch(ctx, gen_init_kernel, dim3(ceil_div(B, 128)), dim3(128), 0, static_cast<cudaStream_t>(stream),
                     ctx->st, d_first, d_budget, B, k_init));
}

int sdv_propose(sdv_ctx *ctx, int drafter, const int32_t *d_table, int table_stride, int B, int max_span,
                int32_t *d_tokens, int32_t *d_row_off, int32_t *d_required, void *stream) {
    if (!ctx || !d_tokens || !d_row_off || !d_required || B <= 0 || B > ctx->c.max_batch || max_span <= 0 ||
        max_span > ctx->c.max_span)
        return SDV_ERR_ARG;
    if (drafter != SDV_DRAFT_NONE && drafter != SDV_DRAFT_NGRAM && drafter != SDV_DRAFT_TABLE) return SDV_ERR_ARG;
    if (drafter == SDV_DRAFT_TABLE && (!d_table || table_stride <= 0)) return SDV_ERR_ARG;
    if (drafter == SDV_DRAFT_NGRAM && ctx->c.ngram_capacity <= 0) return SDV_ERR_UNSUPPORTED;
    const int n_max = ngram_orders(ctx->c);
    const int ng_req = ngram_required(std::min(ctx->ng_min, n_max), n_max, ctx->ng_pmin);
    return rc(launch(ctx, propose_kernel, dim3(1), dim3(256), 0, static_cast<cudaStream_t>(stream), ctx->st, drafter,
                     d_table, table_stride, B, max_span, ng_req, d_tokens, d_row_off, d_required));
}

int sdv_ngram_params(sdv_ctx *ctx, int min_order, float pmin) {
    if (!ctx || min_order < 1 || min_order > ngram_orders(ctx->c) || !(pmin >= 0.f && pmin <= 1.f))
        return SDV_ERR_ARG;
    ctx->ng_min = min_order;
    ctx->ng_pmin = pmin;
    return SDV_OK;
}

int sdv_reset_seq(sdv_ctx *ctx, int b, void *stream) {
    if (!ctx || b < 0 || b >= ctx->c.max_batch) return SDV_ERR_ARG;
    reset_seq_kernel<<<1, 256, 0, static_cast<cudaStream_t>(stream)>>>(ctx->st, b);
    return rc(cudaGetLastError());
}

int sdv_get_status(sdv_ctx *ctx, int32_t *h_status) {
    if (!ctx || !h_status) return SDV_ERR_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return SDV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ctx->st.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDV_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(ctx->st.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SDV_ERR_CUDA;
    *h_status = v;
    return SDV_OK;
}

const char *sdv_status_str(int code) {
    switch (code) {
        case SDV_OK: return "ok";
        case SDV_ERR_ARG: return "invalid argument";
        case SDV_ERR_CAPACITY: return "out of KV capacity";
        case SDV_ERR_CUDA: return "CUDA error";
        case SDV_ERR_DEVICE: return "invalid device input";
        case SDV_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case SDV_ERR_UNSUPPORTED: return "unsupported";
        default: return "unknown status";
    }
}

int sdv_profile_enable(sdv_ctx *ctx, int on) {
    if (!ctx) return SDV_ERR_ARG;
    ctx->profiling = on != 0;
    return SDV_OK;
}

int sdv_profile_read(sdv_ctx *ctx, float *h_ms, int32_t *h_count) {
    if (!ctx || !h_ms || !h_count) return SDV_ERR_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return SDV_ERR_CUDA;
    for (const auto &mk : ctx->ev_marks) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, ctx->ev_pool[mk.second.first], ctx->ev_pool[mk.second.second]) != cudaSuccess)
            return SDV_ERR_CUDA;
        if (mk.first >= 0 && mk.first < 7) {
            h_ms[mk.first] += ms;
            h_count[mk.first] += 1;
        }
    }
    ctx->ev_marks.clear();
    ctx->ev_used = 0;
    return SDV_OK;
}

int sdv_fwd_trace(sdv_ctx *ctx, void *d_buf, size_t bytes) {
    if (!ctx) return SDV_ERR_ARG;
    if (!d_buf) {
        ctx->trace = nullptr;
        ctx->trace_words = 0;
        return SDV_OK;
    }
    if (reinterpret_cast<uintptr_t>(d_buf) % 8) return SDV_ERR_ARG;
    // at least the attention and GEMM regions of the first layer
    if (bytes < kTraceRegionWords * 5 * sizeof(unsigned long long)) return SDV_ERR_ARG;
    ctx->trace = static_cast<unsigned long long *>(d_buf);
    ctx->trace_words = bytes / sizeof(unsigned long long);
    return SDV_OK;
}

int sdv_op_attention(sdv_ctx *ctx, int layer, const void *d_q, const int32_t *d_row_off, const int32_t *d_base,
                     int B, int max_span, void *d_out, void *stream) {
    if (!ctx || !d_q || !d_row_off || !d_base || !d_out || layer < 0 || layer >= ctx->m.n_layers) return SDV_ERR_ARG;
    if (B <= 0 || B > ctx->c.max_batch || max_span <= 0 || max_span > ctx->c.max_span) return SDV_ERR_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int max_rows = ctx->c.max_rows;
    int r = prepare(ctx, nullptr, d_row_off, d_base, B, max_rows, max_span, 0, st);
    if (r) return r;
    return run_attention(ctx, layer, static_cast<const bf16 *>(d_q), 0, static_cast<bf16 *>(d_out), 0, B, max_span, st);
}

}  // extern "C"
