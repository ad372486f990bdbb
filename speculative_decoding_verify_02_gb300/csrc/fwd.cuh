// Persistent verify forward: every decoder layer (QKV, attention, O, gate/up,
// down) and the LM head run inside one cooperative launch of one CTA per SM.
//
// Why: at verify widths (16..128 rows) each projection is a pure weight stream
// (8.04 GB per step for the 4B shape), and a launch per projection pays a
// pipeline fill, an epilogue and an exit every few microseconds. Here the
// weight producer of each CTA never stops: it streams the next phase's weight
// tiles into the shared-memory ring while the current phase's epilogue, its
// cross-CTA reductions and the wait for the phase's inputs are still running.
//
// Work split: a GEMM phase is the list of (output tile, 64-wide k-block)
// units, tile-major; CTA c takes units [c*U/G, (c+1)*U/G). A tile whose units
// span several CTAs is a split tile: each CTA parks its fp32 partial in global
// memory and the last to arrive adds them in CTA order, then runs the tile's
// epilogue. The split depends only on the weight shape and the SM count, so
// a row's result never depends on how many rows share the launch.
//
// Attention: items of (sequence, span-row slice, 128-key chunk, kv head); a
// chunk's partial (m, l, o) is merged with the others of its row slice by the
// last chunk to arrive, in chunk order. Keys are cut by position only.
//
// Phase order: for each layer QKV, ATTN, O, GU, DOWN; then LM. Phase p may
// start reading its inputs once done[p-1] reaches the previous phase's unit
// count (tiles for a GEMM, items for attention); the counters are released
// with a gpu-scope fence and read with acquire loads. Every wait is bounded:
// on a timeout the kernel records SDV_ERR_DEVICE_TIMEOUT, raises a global
// abort flag that every other wait also watches, waits for its own copies in
// flight, frees its TMEM and returns.
//
// Warp roles (384 threads): warps 0-7 epilogue and attention (warps 0-3, one
// per TMEM lane quarter, read the accumulators), warp 8 weight TMA producer,
// warp 9 tcgen05 MMA issuer (and TMEM owner), warp 10 activation TMA producer,
// warp 11 copier (weight tiles, shared -> tensor memory).
#pragma once

#include "attention.cuh"
#include "common.cuh"
#include "gemm.cuh"

namespace sdv {

constexpr int kEpiWarps = 8;                        // epilogue and attention warps (0-7)
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kWarpProducerA = kEpiWarps, kWarpMma = kEpiWarps + 1, kWarpProducerB = kEpiWarps + 2;
constexpr int kWarpCopier = kEpiWarps + 3;
constexpr int kFwdThreads = kEpiThreads + 128;
constexpr int kFwdRows = 32;     // attention query rows (heads x span rows) per item
constexpr int kFwdChunk = 128;   // keys per attention item
constexpr int kFwdSmemLimit = 232448;
constexpr int kFwdMaxHolders = 256;  // CTAs sharing one split tile (at most the grid)

enum FwdPhase : int { FP_QKV = 0, FP_ATTN = 1, FP_O = 2, FP_GU = 3, FP_DOWN = 4, FP_LM = 5 };

struct FwdGemm {
    int tiles, kblocks;
};

struct FwdLayer {
    const bf16 *q_gain, *k_gain;
    const bf16 *ffn_norm;   // gain of the norm before the FFN
    const bf16 *next_norm;  // next layer's attention-norm gain, or the final norm's
};

struct FwdParams {
    const CUtensorMap *tm_w;  // [n_layers * 7 + 1]: per layer wq wk wv wo wg wu wd, then the LM head
    const CUtensorMap *tm_b;  // [3]: norm input, attention output, SwiGLU output (this launch's row width)
    const FwdLayer *layers;
    int n_layers, grid;
    FwdGemm g[5];             // qkv, o, gate/up, down, lm head
    GemmArgs ga[4];           // epilogue arguments per EpiKind; the per-layer fields are patched per phase
    size_t layer_stride;      // KV pool elements per layer
    bf16 *pool;
    bf16 *attn_out;           // [2 planes][rows_cap][nq * D]
    size_t q_plane;           // elements per plane of Q and of the attention output
    // attention items: (b | slice << 16, chunk | n_chunks << 16, L_b, S_b)
    const int4 *items;
    const int *n_items;
    const int *row_off;
    int rps, max_slices;
    int page_shift;           // log2(page size): the persistent path needs a power-of-two page size
    float scale_log2;
    float *att_o;             // [items * nkv][kFwdRows][D]
    float2 *att_ml;           // [items * nkv][kFwdRows]
    int *att_cnt;             // [max_batch][max_slices][nkv]
    // cross-CTA synchronisation
    int *done;                // [5 * n_layers + 1]
    int *tile_cnt;            // [5][tile_stride]
    int tile_stride;
    float *part;              // [2 * grid][rows_cap][128]
    int *abort_flag;
    // split tiles: per plan, at hold + hold_base[i]: [tiles + 1] offsets, then the partial slots of
    // each tile's holders in CTA order (a tile with one holder is not split)
    const int *hold;
    int hold_base[5];
    int ring;                 // weight-ring slots in use (3..the kernel's slots; other values: all)
    // optional timeline: [grid][phases][16] %globaltimer stamps, nullptr when not tracing:
    // 0 inputs ready, 1 last MMA issued, 2 epilogue (or attention) work done, 3 last weight load
    // issued; GEMM epilogue, first segment: 4 accumulator ready, 5 partial parked, 6 split tile's
    // partials loaded; attention, first item: 4 Q copies issued, 5 K/V copies issued, 6 copies
    // landed, 7 softmax and P.V done, 8 partial stored, 9 fenced, 10 arrived, 11 merge fenced,
    // 12 first merge block landed, 13 first merge block written, 14 merge done
    unsigned long long *trace;
};

__device__ __forceinline__ void fwd_stamp(const FwdParams &P, int p, int ev) {
    if (P.trace && p >= 0) P.trace[(static_cast<size_t>(blockIdx.x) * (5 * P.n_layers + 1) + p) * 16 + ev] = globaltimer();
}

// ------------------------------------------------------------------ memory-model helpers
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed_gpu(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void red_release_gpu(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile_i(const int *p) { return *reinterpret_cast<const volatile int *>(p); }
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Make generic-proxy global writes of other CTAs, already acquired, visible to this thread's TMA reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void raise_abort(const FwdParams &P, int *status) {
    set_status(status, SDV_ERR_DEVICE_TIMEOUT);
    atomicExch(P.abort_flag, 1);
}

// try_wait with a suspend-time hint: the thread sleeps until the phase completes or the hint
// runs out, instead of re-issuing the probe (a hot probe loop crowds the shared-memory pipe that
// the epilogue warps need).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// mbarrier wait that also gives up when another CTA has aborted.
__device__ __forceinline__ bool fwd_bar_wait(const FwdParams &P, int *status, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if ((n & 7u) == 7u) {
            if (ld_volatile_i(P.abort_flag)) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                raise_abort(P, status);
                return false;
            }
        }
    }
}

// Wait until *ctr >= target, then acquire; false on timeout or abort. The spin uses relaxed
// loads (an acquire load per poll would disturb the SM's other warps), and one fence orders
// everything after it.
__device__ __forceinline__ bool fwd_count_wait(const FwdParams &P, int *status, const int *ctr, int target) {
    if (ld_relaxed_gpu(ctr) >= target) {
        fence_acq_rel_gpu();
        return true;
    }
    const uint64_t t0 = globaltimer();
    for (;;) {
        __nanosleep(64);
        if (ld_relaxed_gpu(ctr) >= target) {
            fence_acq_rel_gpu();
            return true;
        }
        if (ld_volatile_i(P.abort_flag)) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            raise_abort(P, status);
            return false;
        }
    }
}

// ------------------------------------------------------------------ phases and the work split
__device__ __forceinline__ int fwd_kind(int p, int n_layers) { return p >= 5 * n_layers ? FP_LM : p % 5; }
__device__ __forceinline__ int fwd_gemm_index(int kind) {
    return kind == FP_QKV ? 0 : kind == FP_O ? 1 : kind == FP_GU ? 2 : kind == FP_DOWN ? 3 : 4;
}
__device__ __forceinline__ int fwd_epi(int kind) {
    return kind == FP_QKV ? EPI_QKV : kind == FP_GU ? EPI_SWIGLU : kind == FP_LM ? EPI_LMHEAD : EPI_RESID;
}
__device__ __forceinline__ int fwd_bmap(int kind) { return kind == FP_O ? 1 : kind == FP_DOWN ? 2 : 0; }

// first unit of CTA c, and the CTA that owns unit u, for U units over G CTAs
// (32-bit: the host keeps U * (G + 1) below 2^31)
__device__ __forceinline__ int unit_begin(int c, int U, int G) {
    return static_cast<int>(static_cast<unsigned>(c) * static_cast<unsigned>(U) / static_cast<unsigned>(G));
}
__device__ __forceinline__ int unit_owner(int u, int U, int G) {
    return static_cast<int>((static_cast<unsigned>(u + 1) * static_cast<unsigned>(G) - 1u) / static_cast<unsigned>(U));
}

// This CTA's units of one GEMM phase, cut at tile boundaries into segments.
struct SegRange {
    int KB, u, u1;
    __device__ __forceinline__ SegRange(const FwdGemm &g, int c, int G) {
        KB = g.kblocks;
        const int U = g.tiles * g.kblocks;
        u = unit_begin(c, U, G);
        u1 = unit_begin(c + 1, U, G);
    }
    __device__ __forceinline__ bool next(int &t, int &kb0, int &kb1) {
        if (u >= u1) return false;
        t = u / KB;
        kb0 = u - t * KB;
        const int e = min(u1, (t + 1) * KB);
        kb1 = e - t * KB;
        u = e;
        return true;
    }
};

// The CTAs holding units of tile t, in order: call with cc = -1 to get the first. When there are
// fewer units than CTAs some CTAs hold none, so the holders of a tile need not be consecutive.
__device__ __forceinline__ bool next_holder(int t, int &cc, const FwdGemm &g, int G) {
    const int U = g.tiles * g.kblocks;
    const int u = cc < 0 ? t * g.kblocks : unit_begin(cc + 1, U, G);
    if (u >= (t + 1) * g.kblocks) return false;
    cc = unit_owner(u, U, G);
    return true;
}

// Partial slot of CTA c's segment of tile t: 2c for the CTA's first segment, 2c + 1 for its last.
__device__ __forceinline__ int part_slot(int t, int c, const FwdGemm &g, int G) {
    const int U = g.tiles * g.kblocks;
    return 2 * c + (t == unit_begin(c, U, G) / g.kblocks ? 0 : 1);
}


// ------------------------------------------------------------------ attention items
constexpr int kRegChunks = 8;  // row slices of at most this many chunks merge in registers

// four output columns num / den as hi and lo bf16 planes (8-byte stores)
__device__ __forceinline__ void store_out4(bf16 *out, size_t plane, size_t oi, float4 num, float den) {
    const Bf16Pair p0 = split_bf16(num.x / den), p1 = split_bf16(num.y / den);
    const Bf16Pair p2 = split_bf16(num.z / den), p3 = split_bf16(num.w / den);
    __nv_bfloat162 hi01, hi23, lo01, lo23;
    hi01.x = p0.hi; hi01.y = p1.hi; hi23.x = p2.hi; hi23.y = p3.hi;
    lo01.x = p0.lo; lo01.y = p1.lo; lo23.x = p2.lo; lo23.y = p3.lo;
    uint2 hv, lv;
    hv.x = *reinterpret_cast<uint32_t *>(&hi01);
    hv.y = *reinterpret_cast<uint32_t *>(&hi23);
    lv.x = *reinterpret_cast<uint32_t *>(&lo01);
    lv.y = *reinterpret_cast<uint32_t *>(&lo23);
    *reinterpret_cast<uint2 *>(out + oi) = hv;
    *reinterpret_cast<uint2 *>(out + oi + plane) = lv;
}
template <int D>
struct FwdAttnSmem {
    static constexpr int ROW = D * 2;
    static constexpr int Q_BYTES = 2 * kFwdRows * ROW;  // hi rows 0..31, lo rows 32..63
    static constexpr int KV_BYTES = kFwdChunk * ROW;    // K (or V) of one chunk
    static constexpr int ML_OFF = Q_BYTES + 2 * KV_BYTES;
    static constexpr int BYTES = ML_OFF + 2 * kFwdRows * 8;
    // after the softmax the K/V region holds the two 64-key blocks' fp32 partials [32][D]
    static_assert(2 * KV_BYTES >= 2 * kFwdRows * D * 4, "key-block partials must fit in the K/V region");
};

// One attention item (sequence b, span-row slice, 128-key chunk, kv head g) on warps 0-7.
// Query row j of the slice is span row q0 + j / grp of q-head g * grp + j % grp and
// attends positions <= L_b + q0 + j / grp. Warp w runs query tile w & 1 against 64-key
// block (w >> 1) & 1 for half (w >> 2) of the head dimension (both halves compute the same
// scores); the two blocks merge in shared memory, then the chunk either writes the
// output (a one-chunk row slice) or parks its partial, and the last chunk of the slice
// to arrive merges every chunk in chunk order.
template <int D>
__device__ void fwd_attn_item(const FwdParams &P, int layer, int item, uint8_t *sm, int *page_s, int *last_s,
                              int ph) {
    using S = FwdAttnSmem<D>;
    constexpr int CH = D / 8;
    const GemmArgs &qa = P.ga[EPI_QKV];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nkv = qa.nkv, nq = qa.nq, grp = nq / nkv;
    const int ci = item / nkv, g = item % nkv;
    const int4 wi = P.items[ci];
    const int b = wi.x & 0xffff, qs = wi.x >> 16, ch = wi.y & 0xffff, nch = wi.y >> 16;
    const int L = wi.z, S_b = wi.w;
    const int row0 = P.row_off[b];
    const int q0 = qs * P.rps;
    const int ni = min(S_b - q0, P.rps);
    const int M = grp * ni;
    const int Mpad = (M + 15) & ~15;
    const int k0 = ch * kFwdChunk, k1 = min(k0 + kFwdChunk, L + q0 + ni);
    const int nblk = (k1 - k0 + kAttnKB - 1) / kAttnKB;
    const int page_size = qa.page_size;
    const size_t head_stride = static_cast<size_t>(page_size) * D;
    const bf16 *kv = P.pool + P.layer_stride * layer;

    uint8_t *sQ = sm;
    const uint32_t sK = smem_u32(sm + S::Q_BYTES);
    const uint32_t sV = sK + S::KV_BYTES;
    float *po_s = reinterpret_cast<float *>(sm + S::Q_BYTES);
    float *po2_s = po_s + kFwdRows * D;
    float2 *ml_s = reinterpret_cast<float2 *>(sm + S::ML_OFF);
    float2 *ml2_s = ml_s + kFwdRows;

    for (int e = tid; e < 2 * kFwdRows * CH; e += kEpiThreads) {  // both planes of rows 0..31 (rows >= M zero-filled)
        const int pl = e / (kFwdRows * CH), j = (e / CH) % kFwdRows, c = e % CH;
        const bool valid = j < M;
        const bf16 *src = qa.q_out;
        if (valid) {
            const int r = row0 + q0 + j / grp, h = g * grp + j % grp;
            src = qa.q_out + pl * P.q_plane + (static_cast<size_t>(r) * nq + h) * D + c * 8;
        }
        cp_async16(smem_u32(sQ) + swz<D>(pl * kFwdRows + j, c), src, valid);
    }
    if (tid == 0) fwd_stamp(P, ph, 4);
    const int ps = P.page_shift, pmask = page_size - 1;
    const int pg0 = k0 >> ps, npg = ((k1 - 1) >> ps) - pg0 + 1;
    for (int i = tid; i < npg; i += kEpiThreads) {
        const int slot_idx = pg0 + i;
        page_s[i] = slot_idx < qa.pages_per_seq
                        ? qa.page_table[static_cast<size_t>(b) * qa.pages_per_seq + slot_idx]
                        : -1;
    }
    named_bar_sync(1, kEpiThreads);
    for (int e = tid; e < nblk * kAttnKB * CH; e += kEpiThreads) {
        const int key = e / CH, c = e % CH;
        const int u = k0 + key;
        bool valid = u < k1;
        const bf16 *srcK = kv, *srcV = kv;
        if (valid) {
            const int page = page_s[(u >> ps) - pg0];
            if (page < 0 || page >= qa.n_pages) {
                set_status(qa.status, SDV_ERR_CAPACITY);
                valid = false;
            } else {
                const size_t base = (static_cast<size_t>(page) * 2 * nkv + g) * head_stride +
                                    static_cast<size_t>(u & pmask) * D + c * 8;
                srcK = kv + base;
                srcV = kv + base + static_cast<size_t>(nkv) * head_stride;
            }
        }
        cp_async16(sK + swz<D>(key, c), srcK, valid);
        cp_async16(sV + swz<D>(key, c), srcV, valid);
    }
    cp_async_commit();
    if (tid == 0) fwd_stamp(P, ph, 5);
    cp_async_wait_all();
    named_bar_sync(1, kEpiThreads);
    if (tid == 0) fwd_stamp(P, ph, 6);

    const int mt = warp & 1, blk = (warp >> 1) & 1, dh = warp >> 2;
    const bool active = blk < nblk && mt * 16 < M;
    const int gq = lane >> 2, tq = lane & 3;
    const int jr0 = mt * 16 + gq, jr1 = jr0 + 8;
    const int lim0 = L + q0 + jr0 / grp, lim1 = L + q0 + jr1 / grp;

    float o[D / 16][4];  // this warp's half of the head dimension
#pragma unroll
    for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (active) {
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t qh[4], ql[4];
            {
                const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = ks * 2 + (lane >> 4);
                ldsm_x4(smem_u32(sQ) + swz<D>(row, c), qh[0], qh[1], qh[2], qh[3]);
                ldsm_x4(smem_u32(sQ) + swz<D>(kFwdRows + row, c), ql[0], ql[1], ql[2], ql[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 8; nt += 2) {
                const int i = lane >> 3;
                const int key = blk * kAttnKB + nt * 8 + (i >> 1) * 8 + (lane & 7);
                const int c = ks * 2 + (i & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK + swz<D>(key, c), b0, b1, b2, b3);
                mma_bf16_16816(s[nt], qh, b0, b1);
                mma_bf16_16816(s[nt + 1], qh, b2, b3);
                mma_bf16_16816(s[nt], ql, b0, b1);
                mma_bf16_16816(s[nt + 1], ql, b2, b3);
            }
        }
        const int ubase = k0 + blk * kAttnKB;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int u = ubase + nt * 8 + tq * 2 + e;
                const bool ok0 = u < k1 && u <= lim0, ok1 = u < k1 && u <= lim1;
                s[nt][e] = ok0 ? s[nt][e] * P.scale_log2 : -INFINITY;
                s[nt][2 + e] = ok1 ? s[nt][2 + e] * P.scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                mx1 = fmaxf(mx1, s[nt][2 + e]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        m0 = mx0;
        m1 = mx1;
        const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int nt = 2 * kk + hf;
                const float p0 = exp2f(s[nt][0] - base0), p1 = exp2f(s[nt][1] - base0);
                const float p2 = exp2f(s[nt][2] - base1), p3 = exp2f(s[nt][3] - base1);
                rs0 += p0 + p1;
                rs1 += p2 + p3;
                const Bf16Pair x0 = split_bf16(p0), x1 = split_bf16(p1), x2 = split_bf16(p2), x3 = split_bf16(p3);
                ph[2 * hf] = pack2(x0.hi, x1.hi);
                ph[2 * hf + 1] = pack2(x2.hi, x3.hi);
                pl[2 * hf] = pack2(x0.lo, x1.lo);
                pl[2 * hf + 1] = pack2(x2.lo, x3.lo);
            }
#pragma unroll
            for (int dn = 0; dn < D / 16; dn += 2) {
                const int i = lane >> 3;
                const int key = blk * kAttnKB + kk * 16 + (i & 1) * 8 + (lane & 7);
                const int c = dh * (D / 16) + dn + (i >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sV + swz<D>(key, c), b0, b1, b2, b3);
                mma_bf16_16816(o[dn], ph, b0, b1);
                mma_bf16_16816(o[dn + 1], ph, b2, b3);
                mma_bf16_16816(o[dn], pl, b0, b1);
                mma_bf16_16816(o[dn + 1], pl, b2, b3);
            }
        }
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
        l0 = rs0;
        l1 = rs1;
    }
    named_bar_sync(1, kEpiThreads);  // K/V no longer read: the region now holds the key blocks' partials
    if (tid == 0) fwd_stamp(P, ph, 7);
    if (mt * 16 < Mpad) {
        float *dst = blk == 0 ? po_s : po2_s;
        float2 *mld = blk == 0 ? ml_s : ml2_s;
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
            const int col = (dh * (D / 16) + dn) * 8 + tq * 2;
            *reinterpret_cast<float2 *>(&dst[jr0 * D + col]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(&dst[jr1 * D + col]) = make_float2(o[dn][2], o[dn][3]);
        }
        if (tq == 0 && dh == 0) {
            mld[jr0] = make_float2(m0, l0);
            mld[jr1] = make_float2(m1, l1);
        }
    }
    named_bar_sync(1, kEpiThreads);
    // the two key blocks of a row merge with weights exp2(m_block - max); computed once per row,
    // the merged (m, l) replaces block 0's and the weights replace block 1's
    for (int j = tid; j < Mpad; j += kEpiThreads) {
        const float2 A = ml_s[j], Bp = ml2_s[j];
        const float Mx = fmaxf(A.x, Bp.x);
        const float sa = A.x == -INFINITY ? 0.f : exp2f(A.x - Mx), sb = Bp.x == -INFINITY ? 0.f : exp2f(Bp.x - Mx);
        ml_s[j] = make_float2(Mx, A.y * sa + Bp.y * sb);
        ml2_s[j] = make_float2(sa, sb);
    }
    named_bar_sync(1, kEpiThreads);
    for (int e4 = tid; e4 < Mpad * D / 4; e4 += kEpiThreads) {
        const float2 w = ml2_s[e4 / (D / 4)];
        float4 a4 = reinterpret_cast<float4 *>(po_s)[e4];
        const float4 b4 = reinterpret_cast<const float4 *>(po2_s)[e4];
        a4.x = a4.x * w.x + b4.x * w.y;
        a4.y = a4.y * w.x + b4.y * w.y;
        a4.z = a4.z * w.x + b4.z * w.y;
        a4.w = a4.w * w.x + b4.w * w.y;
        reinterpret_cast<float4 *>(po_s)[e4] = a4;
    }
    named_bar_sync(1, kEpiThreads);

    bf16 *out = P.attn_out;
    if (nch == 1) {
        for (int e = tid; e < M * D; e += kEpiThreads) {
            const int j = e / D, d = e % D;
            const int r = row0 + q0 + j / grp, h = g * grp + j % grp;
            const size_t oi = (static_cast<size_t>(r) * nq + h) * D + d;
            const Bf16Pair pr = split_bf16(po_s[e] / ml_s[j].y);
            out[oi] = pr.hi;
            out[oi + P.q_plane] = pr.lo;
        }
        return;
    }
    const size_t slot = static_cast<size_t>(item);
    {
        const float4 *src4 = reinterpret_cast<const float4 *>(po_s);
        float4 *dst4 = reinterpret_cast<float4 *>(P.att_o + slot * kFwdRows * D);
        for (int e = tid; e < M * D / 4; e += kEpiThreads) dst4[e] = src4[e];
    }
    for (int j = tid; j < M; j += kEpiThreads) P.att_ml[slot * kFwdRows + j] = ml_s[j];
    if (tid == 0) fwd_stamp(P, ph, 8);
    named_bar_sync(1, kEpiThreads);  // every thread's partial is written; thread 0's acq_rel atomic releases them all
    if (tid == 0) fwd_stamp(P, ph, 9);
    if (tid == 0) {
        int *cnt = &P.att_cnt[(static_cast<size_t>(b) * P.max_slices + qs) * nkv + g];
        const int last = atom_add_acq_rel_gpu(cnt, 1) == nch - 1;
        if (last) *cnt = 0;
        *last_s = last;
        fwd_stamp(P, ph, 10);
    }
    named_bar_sync(1, kEpiThreads);  // thread 0's acquire covers the reads below
    if (!*last_s) return;
    if (tid == 0) fwd_stamp(P, ph, 11);
    // every chunk's partial for a block of rows, copied into shared memory in one burst, then merged
    // in chunk order: Mx = max m, out = sum exp2(m - Mx) o / sum exp2(m - Mx) l
    const size_t first = static_cast<size_t>(ci - ch) * nkv + g;  // the chunks of a slice are consecutive items
    if (nch <= kRegChunks) {
        // few chunks: one pass computes each row's chunk weights exp2(m - Mx) and denominator into
        // shared memory (reusing the partial region) while every thread already has its o loads in
        // flight; then each thread combines its columns in chunk order
        constexpr int PER = kFwdRows * (D / 4) / kEpiThreads;  // float4 columns per thread
        constexpr int GRP = PER < 2 ? PER : 2;                  // columns whose loads are in flight together
        float *wsc = reinterpret_cast<float *>(sm);  // [kFwdRows][kRegChunks + 1]: weights, then denominator
        for (int i0 = 0; i0 < PER; i0 += GRP) {
            float4 o4[GRP][kRegChunks];
#pragma unroll
            for (int i = 0; i < GRP; ++i) {
                const int e4 = tid + (i0 + i) * kEpiThreads, j = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
#pragma unroll
                for (int cc = 0; cc < kRegChunks; ++cc)
                    if (cc < nch && j < M)
                        o4[i][cc] = __ldcg(reinterpret_cast<const float4 *>(
                            P.att_o + ((first + static_cast<size_t>(cc) * nkv) * kFwdRows + j) * D + d));
            }
            if (i0 == 0) {
                if (tid < M) {
                    float2 ml[kRegChunks];
#pragma unroll
                    for (int cc = 0; cc < kRegChunks; ++cc)
                        if (cc < nch) ml[cc] = __ldcg(&P.att_ml[(first + static_cast<size_t>(cc) * nkv) * kFwdRows + tid]);
                    float Mx = -INFINITY;
#pragma unroll
                    for (int cc = 0; cc < kRegChunks; ++cc)
                        if (cc < nch) Mx = fmaxf(Mx, ml[cc].x);
                    float den = 0.f;
#pragma unroll
                    for (int cc = 0; cc < kRegChunks; ++cc)
                        if (cc < nch) {
                            const float sc = ml[cc].x == -INFINITY ? 0.f : exp2f(ml[cc].x - Mx);
                            wsc[tid * (kRegChunks + 1) + cc] = sc;
                            den += sc * ml[cc].y;
                        }
                    wsc[tid * (kRegChunks + 1) + kRegChunks] = den;
                }
                named_bar_sync(1, kEpiThreads);
            }
#pragma unroll
            for (int i = 0; i < GRP; ++i) {
                const int e4 = tid + (i0 + i) * kEpiThreads, j = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
                if (j >= M) continue;
                float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int cc = 0; cc < kRegChunks; ++cc)
                    if (cc < nch) {
                        const float sc = wsc[j * (kRegChunks + 1) + cc];
                        num.x += sc * o4[i][cc].x;
                        num.y += sc * o4[i][cc].y;
                        num.z += sc * o4[i][cc].z;
                        num.w += sc * o4[i][cc].w;
                    }
                store_out4(out, P.q_plane, (static_cast<size_t>(row0 + q0 + j / grp) * nq + g * grp + j % grp) * D + d,
                           num, wsc[j * (kRegChunks + 1) + kRegChunks]);
            }
        }
        if (tid == 0) fwd_stamp(P, ph, 14);
        return;
    }
    const int rows_fit = (S::BYTES - 16) / (nch * (D * 4 + 12) + 4);
    if (rows_fit < 1) {  // more chunks than shared memory holds: merge straight from global memory
        for (int e = tid; e < M * D; e += kEpiThreads) {
            const int j = e / D, d = e % D;
            float Mx = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) Mx = fmaxf(Mx, __ldcg(&P.att_ml[(first + cc * nkv) * kFwdRows + j].x));
            float num = 0.f, den = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
                const size_t sl = first + static_cast<size_t>(cc) * nkv;
                const float2 ml = __ldcg(&P.att_ml[sl * kFwdRows + j]);
                const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
                den += sc * ml.y;
                num += sc * __ldcg(&P.att_o[(sl * kFwdRows + j) * D + d]);
            }
            const int r = row0 + q0 + j / grp, h = g * grp + j % grp;
            const size_t oi = (static_cast<size_t>(r) * nq + h) * D + d;
            const Bf16Pair pr = split_bf16(num / den);
            out[oi] = pr.hi;
            out[oi + P.q_plane] = pr.lo;
        }
        return;
    }
    const int rc = min(M, rows_fit);
    float *so = reinterpret_cast<float *>(sm);                                   // [nch][rc][D]
    float2 *sml = reinterpret_cast<float2 *>(so + static_cast<size_t>(nch) * rc * D);  // [nch][rc]
    float *ssc = reinterpret_cast<float *>(sml + static_cast<size_t>(nch) * rc);     // [nch][rc] chunk weights
    float *sden = ssc + static_cast<size_t>(nch) * rc;                               // [rc]
    for (int j0 = 0; j0 < M; j0 += rc) {
        const int nr = min(rc, M - j0);
        for (int cc = 0; cc < nch; ++cc) {
            const float *src = P.att_o + ((first + static_cast<size_t>(cc) * nkv) * kFwdRows + j0) * D;
            for (int idx = tid; idx < nr * (D / 4); idx += kEpiThreads)
                cp_async16(smem_u32(so + (cc * nr) * D + idx * 4), src + idx * 4, true);
        }
        cp_async_commit();
        for (int e = tid; e < nch * nr; e += kEpiThreads) {
            const int cc = e / nr, rr = e - cc * nr;
            sml[e] = __ldcg(&P.att_ml[(first + static_cast<size_t>(cc) * nkv) * kFwdRows + j0 + rr]);
        }
        named_bar_sync(1, kEpiThreads);
        // per row: Mx = max m, weight of chunk cc = exp2(m_cc - Mx), denominator = sum weight * l
        for (int rr = tid; rr < nr; rr += kEpiThreads) {
            float Mx = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) Mx = fmaxf(Mx, sml[cc * nr + rr].x);
            float den = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
                const float2 ml = sml[cc * nr + rr];
                const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
                ssc[cc * nr + rr] = sc;
                den += sc * ml.y;
            }
            sden[rr] = den;
        }
        cp_async_wait_all();
        named_bar_sync(1, kEpiThreads);
        if (tid == 0 && j0 == 0) fwd_stamp(P, ph, 12);
        // out = sum over chunks, in order, of weight * o, over the denominator; four columns a thread
        for (int e4 = tid; e4 < nr * (D / 4); e4 += kEpiThreads) {
            const int rr = e4 / (D / 4), d = (e4 % (D / 4)) * 4, j = j0 + rr;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int cc = 0; cc < nch; ++cc) {
                const float sc = ssc[cc * nr + rr];
                const float4 o4 = *reinterpret_cast<const float4 *>(so + (cc * nr + rr) * D + d);
                num.x += sc * o4.x;
                num.y += sc * o4.y;
                num.z += sc * o4.z;
                num.w += sc * o4.w;
            }
            store_out4(out, P.q_plane, (static_cast<size_t>(row0 + q0 + j / grp) * nq + g * grp + j % grp) * D + d,
                       num, sden[rr]);
        }
        named_bar_sync(1, kEpiThreads);
        if (tid == 0 && j0 == 0) fwd_stamp(P, ph, 13);
    }
    if (tid == 0) fwd_stamp(P, ph, 14);
}


// ------------------------------------------------------------------ the kernel
// Shared memory: a ring of SA weight tiles (16 KB, TMA destination), then one region that
// attention uses whole during an attention phase and that otherwise holds a 64 KB ring of SB
// activation tiles followed by the epilogue's staging area. (Attention runs only after every
// activation tile of the phase before it was consumed, and the next phase's activations load only
// after every attention item is done.) Tensor memory (all 512 columns): two accumulators of NC
// columns, then NT weight-tile slots of 32 columns that the MMA reads its A operand from. A weight
// tile moves shared -> tensor memory (tcgen05.cp) as soon as it lands, so the shared slot turns
// over at copy speed and up to NT tiles wait on chip for their activations.
template <int N, int D>
struct FwdShape {
    using GS = GemmShape<N>;
    static constexpr int A_TILE = GS::A_BYTES;   // 16 KB
    static constexpr int B_TILE = GS::B_BYTES;   // hi and lo planes, N rows x 64
    static constexpr int TOTAL = kFwdSmemLimit - 1024 - 3072;  // alignment slack, static shared memory
    static constexpr int SA = 7;
    static constexpr int X_OFF = SA * A_TILE;
    static constexpr int X_BYTES = (TOTAL - X_OFF) & ~1023;
    static constexpr int B_RING = 65536;
    static constexpr int SB = B_RING / B_TILE;
    static constexpr int B_OFF = X_OFF;
    static constexpr int STAGE_OFF = X_OFF + B_RING;
    static constexpr int STAGE_BYTES = X_BYTES - B_RING;  // epilogue staging
    static constexpr int ATT_OFF = X_OFF;
    // An accumulator holds the hi-plane product in columns [0, N) and the lo-plane product in
    // [N, 2N); the epilogue adds them. Up to N = 64 one MMA of width 2N covers both planes (the
    // activation tile stores the lo rows right after the hi rows), which halves the MMA count per
    // weight byte; at N = 128 each plane is its own MMA and a single accumulator fits beside the
    // weight slots.
    static constexpr bool COMBINED = N <= 64;
    static constexpr int NC = 2 * N;                  // TMEM columns per accumulator
    static constexpr int ACC = COMBINED ? 2 : 1;      // accumulators (ping-pong between segments)
    static constexpr uint32_t IDESC = idesc_bf16(128, COMBINED ? 2 * N : N);
    static constexpr int TMEM_COLS = 512;
    static constexpr int NT = (TMEM_COLS - ACC * NC) / 32;
    static constexpr int SMEM_BYTES = X_OFF + X_BYTES + 1024;
    static_assert(FwdAttnSmem<D>::BYTES <= X_BYTES, "attention must fit the shared region");
    static_assert(STAGE_BYTES >= 32 * 128 * 4, "staging holds 32 rows of a tile");
    static_assert(SB >= 2 && NT >= 4, "pipeline too shallow");
};

// tcgen05 forms for a weight tile staged in tensor memory: copy 128 rows x 32 bytes (one 16-wide
// k slice) from shared memory through a matrix descriptor, and an MMA that reads A from TMEM.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Shared state the epilogue warps use.
struct FwdEpiCtx {
    uint64_t *acc_full, *acc_empty;
    EpiSmem *es;
    float *stage;     // staging region (shared with attention)
    int *flag, *last;
    uint32_t tmem;
    int *status;
    int R, rows_cap, c, G, stage_bytes, nc, n, acc_slots;
};

// Count one finished tile of phase p; the last tile of the LM head publishes the argmax.
template <int EK>
__device__ __forceinline__ void fwd_tile_done(const FwdParams &P, const FwdEpiCtx &E, int p, int tiles) {
    const int tid = threadIdx.x;
    named_bar_sync(1, kEpiThreads);
    if (tid == 0) {
        const int prev = atom_add_acq_rel_gpu(&P.done[p], 1);
        *E.last = EK == EPI_LMHEAD && prev == tiles - 1;
    }
    named_bar_sync(1, kEpiThreads);
    if constexpr (EK == EPI_LMHEAD) {
        if (*E.last) {  // every tile's row maxima are in: publish the argmax
            const GemmArgs &a = P.ga[EK];
            for (int r = tid; r < E.R; r += kEpiThreads) {
                const unsigned long long k = atomicAdd(&a.keys[r], 0ull);
                a.argmax_out[r] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
            }
        }
    }
}

// The epilogue warps' part of one GEMM phase of kind EK. First every segment this CTA holds,
// in order: a whole tile goes accumulator -> staging -> a warp per row; a split tile's
// partial is parked in global memory and the holder's arrival counted. Then, for the split
// tiles where this CTA arrived last, every holder's partial (and, for a residual epilogue,
// the old residual rows) is copied into shared memory in one burst and added in holder (CTA)
// order. Returns false on abort.
template <int EK>
__device__ bool fwd_gemm_epi(const FwdParams &P, const FwdEpiCtx &E, const EpiLayer &el, int p, int gi, int &q,
                             bool first_phase_seg_stamp) {
    const GemmArgs &a = P.ga[EK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = E.R, rows_cap = E.rows_cap, c = E.c, G = E.G;
    EpiSmem &es = *E.es;
    if constexpr (EK != EPI_RESID) {  // rstd of the RMSNorm feeding this GEMM; partial sums in tile order
        if (tid < R) {
            float sum = 0.f;
            for (int t0 = 0; t0 < a.ss_tiles; t0 += 8) {
                float v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = t0 + i < a.ss_tiles ? __ldcg(&a.ss_in[static_cast<size_t>(t0 + i) * rows_cap + tid]) : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (t0 + i < a.ss_tiles) sum += v[i];
            }
            es.rstd[tid] = rsqrtf(sum / static_cast<float>(a.hidden) + a.eps);
        }
        named_bar_sync(1, kEpiThreads);
    }
    const FwdGemm gm = P.g[gi];
    const int *hoff = P.hold + P.hold_base[gi];
    const int *hslot = hoff + gm.tiles + 1;
    const int my_first_tile = unit_begin(c, gm.tiles * gm.kblocks, G) / gm.kblocks;
    SegRange sr(gm, c, G);
    int t, kb0, kb1;
    bool first_seg = first_phase_seg_stamp;
    int pend_t[2], npend = 0;  // split tiles this CTA reduces (at most its first and last segment)
    while (sr.next(t, kb0, kb1)) {
        const int acc = q % E.acc_slots;
        if (tid == 0) *E.flag = fwd_bar_wait(P, E.status, &E.acc_full[acc], (q / E.acc_slots) & 1);
        named_bar_sync(1, kEpiThreads);
        const int go = *E.flag;
        named_bar_sync(1, kEpiThreads);
        if (!go) return false;
        if (tid == 0 && first_seg) fwd_stamp(P, p, 4);
        tc_fence_after();
        const int h0 = __ldg(&hoff[t]), nh = __ldg(&hoff[t + 1]) - h0;
        const uint32_t tacc = E.tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>(acc * E.nc);
        float v[32];
        if (nh == 1) {
            for (int c0 = 0; c0 < R; c0 += 32) {
                if (warp < 4) {
                    acc_load(tacc, c0, E.n, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < R) E.stage[j * 128 + tid] = v[j];
                }
                named_bar_sync(1, kEpiThreads);
                for (int r = c0 + warp; r < min(R, c0 + 32); r += kEpiWarps) {
                    float x[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[i] = E.stage[(r - c0) * 128 + lane + 32 * i];
                    epi_row<EK>(a, el, es, t, r, lane, x);
                }
                named_bar_sync(1, kEpiThreads);
            }
            tc_fence_before();
            named_bar_sync(1, kEpiThreads);
            if (tid == 0) mbar_arrive(&E.acc_empty[acc]);
            fwd_tile_done<EK>(P, E, p, gm.tiles);
        } else {
            const int my_slot = 2 * c + (t == my_first_tile ? 0 : 1);
            float *pp = P.part + static_cast<size_t>(my_slot) * rows_cap * 128;
            if (warp < 4)
                for (int c0 = 0; c0 < R; c0 += 32) {
                    acc_load(tacc, c0, E.n, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < R) pp[static_cast<size_t>(c0 + j) * 128 + tid] = v[j];
                }
            tc_fence_before();
            named_bar_sync(1, kEpiThreads);  // thread 0's acq_rel atomic releases every thread's partial
            if (tid == 0) {
                mbar_arrive(&E.acc_empty[acc]);
                const int last = atom_add_acq_rel_gpu(&P.tile_cnt[gi * P.tile_stride + t], 1) == nh - 1;
                if (last) P.tile_cnt[gi * P.tile_stride + t] = 0;
                *E.last = last;
                if (first_seg) fwd_stamp(P, p, 5);
            }
            named_bar_sync(1, kEpiThreads);
            if (*E.last) pend_t[npend++] = t;
            named_bar_sync(1, kEpiThreads);
        }
        ++q;
        first_seg = false;
    }
    for (int k = 0; k < npend; ++k) {  // thread 0's acquire (the arrival atomic) covers these reads
        t = pend_t[k];
        const int h0 = __ldg(&hoff[t]), nh = __ldg(&hoff[t + 1]) - h0;
        constexpr int extra = EK == EPI_RESID ? 1 : 0;  // the old residual rows ride along
        const int rc = min(32, E.stage_bytes / ((nh + extra) * 512));
        for (int r0 = 0; r0 < R; r0 += rc) {
            const int nr = min(rc, R - r0);
            for (int h = 0; h < nh; ++h) {
                const float *src = P.part + (static_cast<size_t>(__ldg(&hslot[h0 + h])) * rows_cap + r0) * 128;
                for (int idx = tid; idx < nr * 32; idx += kEpiThreads)
                    cp_async16(smem_u32(E.stage + (h * nr + (idx >> 5)) * 128 + (idx & 31) * 4),
                               src + (idx >> 5) * 128 + (idx & 31) * 4, true);
            }
            if constexpr (EK == EPI_RESID) {
                for (int idx = tid; idx < nr * 32; idx += kEpiThreads) {
                    const int rr = idx >> 5, q4 = idx & 31;
                    const bool in = t * 128 + q4 * 4 < a.n_out;  // features past the hidden size read as 0
                    cp_async16(smem_u32(E.stage + (nh * nr + rr) * 128 + q4 * 4),
                               in ? a.x + static_cast<size_t>(r0 + rr) * a.hidden + t * 128 + q4 * 4 : a.x, in);
                }
            }
            cp_async_commit();
            cp_async_wait_all();
            named_bar_sync(1, kEpiThreads);
            if (tid == 0 && r0 == 0 && k == 0 && first_phase_seg_stamp) fwd_stamp(P, p, 6);
            for (int r = r0 + warp; r < r0 + nr; r += kEpiWarps) {
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                for (int h = 0; h < nh; ++h) {
                    const float *src = E.stage + (h * nr + (r - r0)) * 128 + lane;
#pragma unroll
                    for (int i = 0; i < 4; ++i) x[i] += src[32 * i];
                }
                if constexpr (EK == EPI_RESID)
                    epi_resid_row(a, el, t, r, lane, x, E.stage + (nh * nr + (r - r0)) * 128);
                else
                    epi_row<EK>(a, el, es, t, r, lane, x);
            }
            named_bar_sync(1, kEpiThreads);
        }
        fwd_tile_done<EK>(P, E, p, gm.tiles);
    }
    return true;
}

// weight tensor maps of phase p: wq wk wv | wo | wg wu | wd | lm
__device__ __forceinline__ const CUtensorMap *fwd_wmap(const FwdParams &P, int kind, int layer) {
    if (kind == FP_LM) return P.tm_w + 7 * P.n_layers;
    const int j = kind == FP_QKV ? 0 : kind == FP_O ? 3 : kind == FP_GU ? 4 : 6;
    return P.tm_w + 7 * layer + j;
}

// Ring slot and phase parity of a role's next k-block, advanced without division.
struct RingPos {
    int s = 0, n = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next(int nst) {
        ++n;
        if (++s == nst) {
            s = 0;
            ph ^= 1u;
        }
    }
    // wait (bounded) until the copies of the last nst k-blocks issued on `full` have landed
    __device__ __forceinline__ void drain(uint64_t *full, int nst) const {
        for (int j = n > nst ? n - nst : 0; j < n; ++j) mbar_wait(&full[j % nst], (j / nst) & 1);
    }
};

// units the phase's consumers wait for
__device__ __forceinline__ int fwd_target(const FwdParams &P, int kind) {
    if (kind == FP_ATTN) return *P.n_items * P.ga[EPI_QKV].nkv;
    return P.g[fwd_gemm_index(kind)].tiles;
}

template <int N, int D>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams P) {
    using F = FwdShape<N, D>;
    using GS = GemmShape<N>;
    constexpr int SA = F::SA, SB = F::SB, NT = F::NT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sB = smem + F::B_OFF;
    uint8_t *att = smem + F::ATT_OFF;
    uint8_t *stage = smem + F::STAGE_OFF;
    __shared__ __align__(8) uint64_t fullA[SA], emptyA[SA], fullB[SB], emptyB[SB], tfree[NT], tcopied[NT];
    __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], fin_bar, fin_bar2;
    __shared__ uint32_t tmem_s;
    __shared__ EpiSmem es;
    __shared__ int page_s[kFwdChunk + 1];
    __shared__ int flag_s, last_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int c = blockIdx.x, G = P.grid, nL = P.n_layers;
    const int n_ph = 5 * nL + 1;
    const int nsa = P.ring >= 3 && P.ring <= SA ? P.ring : SA;  // weight-ring slots in use
    int *status = P.ga[EPI_QKV].status;

    if (tid == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(&fullA[s], 1);
            mbar_init(&emptyA[s], 1);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(&fullB[s], 1);
            mbar_init(&emptyB[s], 1);
        }
        for (int s = 0; s < NT; ++s) {
            mbar_init(&tfree[s], 1);
            mbar_init(&tcopied[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 1);
        }
        mbar_init(&fin_bar, 1);
        mbar_init(&fin_bar2, 1);
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&tmem_s, F::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    pdl_trigger();
    pdl_wait();

    if (warp == kWarpProducerA) {
        // ---------------- weight producer: never waits on another CTA. It loads the weight ring in
        // consumption order; the tensor maps and row coordinate of a segment are resolved once per
        // segment.
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            RingPos rp;
            bool ok = true;
            for (int p = 0; p < n_ph && ok; ++p) {
                const int kind = fwd_kind(p, nL);
                if (kind == FP_ATTN) continue;
                const int ek = fwd_epi(kind);
                const CUtensorMap *tw = fwd_wmap(P, kind, p / 5);
                const GemmArgs &ga = P.ga[ek];
                SegRange sr(P.g[fwd_gemm_index(kind)], c, G);
                int t, kb0, kb1;
                while (ok && sr.next(t, kb0, kb1)) {
                    const CUtensorMap *m0 = tw, *m1 = nullptr;
                    int row = t * 128;
                    if (ek == EPI_QKV) {
                        if (t >= ga.q_tiles + ga.k_tiles) {
                            m0 = tw + 2;
                            row = (t - ga.q_tiles - ga.k_tiles) * 128;
                        } else if (t >= ga.q_tiles) {
                            m0 = tw + 1;
                            row = (t - ga.q_tiles) * 128;
                        }
                    } else if (ek == EPI_SWIGLU) {  // rows 0-63 gate, rows 64-127 the matching up features
                        m1 = tw + 1;
                        row = t * 64;
                    }
                    for (int kc = kb0 * 64; kc < kb1 * 64; kc += 64) {
                        if (!fwd_bar_wait(P, status, &emptyA[rp.s], rp.ph ^ 1)) {
                            ok = false;
                            break;
                        }
                        uint8_t *dst = smem + rp.s * F::A_TILE;
                        mbar_arrive_expect_tx(&fullA[rp.s], F::A_TILE);
                        tma_load_2d_hint(dst, m0, &fullA[rp.s], kc, row, pol);
                        if (m1) tma_load_2d_hint(dst + F::A_TILE / 2, m1, &fullA[rp.s], kc, row, pol);
                        rp.next(nsa);
                    }
                }
                fwd_stamp(P, p, 3);
            }
            rp.drain(fullA, nsa);  // own copies in flight
        }
        __syncwarp();
    } else if (warp == kWarpProducerB) {
        // ---------------- activation producer: waits for the previous phase, then loads B
        if (lane == 0) {
            RingPos rp;
            bool ok = true;
            for (int p = 0; p < n_ph && ok; ++p) {
                const int kind = fwd_kind(p, nL);
                if (kind == FP_ATTN) continue;
                if (p > 0) {
                    if (!fwd_count_wait(P, status, &P.done[p - 1], fwd_target(P, fwd_kind(p - 1, nL)))) break;
                    fence_proxy_async_global();
                }
                fwd_stamp(P, p, 0);
                const CUtensorMap *tb = P.tm_b + fwd_bmap(kind);
                SegRange sr(P.g[fwd_gemm_index(kind)], c, G);
                int t, kb0, kb1;
                while (ok && sr.next(t, kb0, kb1)) {
                    for (int kc = kb0 * 64; kc < kb1 * 64; kc += 64) {
                        if (!fwd_bar_wait(P, status, &emptyB[rp.s], rp.ph ^ 1)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&fullB[rp.s], F::B_TILE);
                        tma_load_3d(sB + rp.s * F::B_TILE, tb, &fullB[rp.s], kc, 0, 0);
                        rp.next(SB);
                    }
                }
            }
            rp.drain(fullB, SB);
        }
        __syncwarp();
    } else if (warp == kWarpCopier) {
        // ---------------- copier: each landed weight tile moves into the next TMEM slot once the
        // MMAs that last read that slot are done; the shared slot is free as soon as the copy is.
        // It never waits on activations, so across a phase hand-off the weights keep streaming.
        if (lane == 0) {
            int total = 0;  // this CTA's k-blocks over every GEMM phase
            for (int p = 0; p < n_ph; ++p) {
                const int kind = fwd_kind(p, nL);
                if (kind == FP_ATTN) continue;
                const FwdGemm &g = P.g[fwd_gemm_index(kind)];
                const int U = g.tiles * g.kblocks;
                total += unit_begin(c + 1, U, G) - unit_begin(c, U, G);
            }
            const uint32_t sa0 = smem_u32(smem), tA = tmem + F::ACC * F::NC;
            RingPos ca, ta;
            for (int it = 0; it < total; ++it) {
                if (!fwd_bar_wait(P, status, &fullA[ca.s], ca.ph) || !fwd_bar_wait(P, status, &tfree[ta.s], ta.ph ^ 1))
                    break;
                tc_fence_after();
                const uint64_t ad = sw128_desc(sa0 + ca.s * F::A_TILE);
                const uint32_t dst = tA + ta.s * 32;
#pragma unroll
                for (int k = 0; k < 4; ++k) tc_cp_128x256b(dst + 8 * k, ad + 2 * k);
                umma_commit(&tcopied[ta.s]);
                umma_commit(&emptyA[ca.s]);
                ca.next(nsa);
                ta.next(NT);
            }
            umma_commit(&fin_bar);  // every copy issued above has completed once this fires
            mbar_wait(&fin_bar, 0);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---------------- MMA issuer: A from the TMEM slot the copier filled, B from the
        // activation ring; two TMEM accumulators, one per segment in flight
        if (lane == 0) {
            const uint32_t sb0 = smem_u32(sB), tA = tmem + F::ACC * F::NC;
            RingPos mt, mb;
            int q = 0;
            bool ok = true;
            for (int p = 0; p < n_ph && ok; ++p) {
                const int kind = fwd_kind(p, nL);
                if (kind == FP_ATTN) continue;
                SegRange sr(P.g[fwd_gemm_index(kind)], c, G);
                int t, kb0, kb1;
                while (ok && sr.next(t, kb0, kb1)) {
                    const int acc = q % F::ACC, use = q / F::ACC;
                    if (use >= 1 && !fwd_bar_wait(P, status, &acc_empty[acc], (use - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(acc * F::NC);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!fwd_bar_wait(P, status, &tcopied[mt.s], mt.ph) ||
                            !fwd_bar_wait(P, status, &fullB[mb.s], mb.ph)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_t = tA + mt.s * 32;
                        const uint64_t bh = sw128_desc(sb0 + mb.s * F::B_TILE);
                        const uint64_t bl = sw128_desc(sb0 + mb.s * F::B_TILE + GS::B_PLANE);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
                            if constexpr (F::COMBINED) {  // both planes: rows 0..N-1 hi, N..2N-1 lo
                                umma_bf16_tmem_a(d, a_t + 8 * k, bh + 2 * k, F::IDESC, accum);
                            } else {
                                umma_bf16_tmem_a(d, a_t + 8 * k, bh + 2 * k, F::IDESC, accum);
                                umma_bf16_tmem_a(d + N, a_t + 8 * k, bl + 2 * k, F::IDESC, accum);
                            }
                        }
                        umma_commit(&emptyB[mb.s]);
                        umma_commit(&tfree[mt.s]);
                        mt.next(NT);
                        mb.next(SB);
                    }
                    if (!ok) break;
                    umma_commit(&acc_full[acc]);
                    ++q;
                }
                fwd_stamp(P, p, 1);
            }
            umma_commit(&fin_bar2);  // every MMA issued above has completed once this fires
            mbar_wait(&fin_bar2, 0);
        }
        __syncwarp();
    } else {
        // ---------------- warps 0-7: epilogues and attention
        int R = *P.ga[EPI_QKV].nrows;
        if (R > N) {
            if (tid == 0) set_status(status, SDV_ERR_ARG);
            R = N;
        }
        const int rows_cap = P.ga[EPI_QKV].rows_cap;
        FwdEpiCtx E;
        E.acc_full = acc_full;
        E.acc_empty = acc_empty;
        E.es = &es;
        E.stage = reinterpret_cast<float *>(stage);
        E.flag = &flag_s;
        E.last = &last_s;
        E.tmem = tmem;
        E.status = status;
        E.R = R;
        E.rows_cap = rows_cap;
        E.c = c;
        E.G = G;
        E.stage_bytes = F::STAGE_BYTES;
        E.nc = F::NC;
        E.n = N;
        E.acc_slots = F::ACC;
        int q = 0;
        for (int p = 0; p < n_ph; ++p) {
            const int kind = fwd_kind(p, nL), layer = p / 5;
            if (p > 0) {  // the previous phase's outputs, and transitively every earlier phase's
                if (tid == 0) flag_s = fwd_count_wait(P, status, &P.done[p - 1], fwd_target(P, fwd_kind(p - 1, nL)));
                named_bar_sync(1, kEpiThreads);
                const int go = flag_s;
                named_bar_sync(1, kEpiThreads);  // every thread has read the flag before it is reused
                if (!go) break;
            }
            if (kind == FP_ATTN) {
                if (tid == 0) fwd_stamp(P, p, 0);
                const int n_it = fwd_target(P, FP_ATTN);
                for (int i = c; i < n_it; i += G) {
                    fwd_attn_item<D>(P, layer, i, att, page_s, &last_s, i == c ? p : -1);
                    named_bar_sync(1, kEpiThreads);
                    if (tid == 0) red_release_gpu(&P.done[p], 1);
                }
                if (tid == 0) fwd_stamp(P, p, 2);
                continue;
            }
            const int gi = fwd_gemm_index(kind);
            EpiLayer el{nullptr, nullptr, nullptr, nullptr};
            bool ok;
            if (kind == FP_QKV) {
                el.q_gain = P.layers[layer].q_gain;
                el.k_gain = P.layers[layer].k_gain;
                el.kv_layer = P.pool + P.layer_stride * layer;
                ok = fwd_gemm_epi<EPI_QKV>(P, E, el, p, gi, q, true);
            } else if (kind == FP_O || kind == FP_DOWN) {
                el.g_next = kind == FP_O ? P.layers[layer].ffn_norm : P.layers[layer].next_norm;
                ok = fwd_gemm_epi<EPI_RESID>(P, E, el, p, gi, q, true);
            } else if (kind == FP_GU) {
                ok = fwd_gemm_epi<EPI_SWIGLU>(P, E, el, p, gi, q, true);
            } else {
                ok = fwd_gemm_epi<EPI_LMHEAD>(P, E, el, p, gi, q, true);
            }
            if (!ok) break;
            if (tid == 0) fwd_stamp(P, p, 2);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, F::TMEM_COLS);
    }
}

}  // namespace sdv
