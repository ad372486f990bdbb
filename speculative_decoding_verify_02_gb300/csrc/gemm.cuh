// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05), used for
// every dense projection of the verify forward: Y[rows][out] = X[rows][in] . W[out][in]^T.
//
// The verify span has few rows (K+1 per sequence, <= 128 in all), so the weight
// matrix is the tcgen05 A operand (M = 128 output features per tile, streamed
// from HBM by TMA with 128-byte swizzle) and the activations are the B operand
// (N = rows padded to 16/32/64/128, read from L2). The accumulator sits in
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
    int n_out;                         // valid output features (ffn for SwiGLU)
    int rows_cap;                      // row stride of partial / ss buffers
    const int *nrows;                  // device: rows present (R)
    int *status;
    // rstd of the RMSNorm feeding this GEMM (QKV, SwiGLU, LM head): from sum-of-squares parts
    const float *ss_in;
    int ss_tiles, hidden;
    float eps;
    // split-K
    float *partial;
    int *counters;
    int part_stride;                   // features per partial row (tiles * 128)
    // QKV epilogue
    int nq, nkv, D, q_tiles, k_tiles, qk_norm;
    const bf16 *q_gain, *k_gain;
    const float2 *rope;                // [positions][D/2] (cos, sin)
    int rope_rows;
    const int *row_seq, *row_pos, *page_table;
    int pages_per_seq, page_size, n_pages;
    bf16 *q_out, *kv_layer;
    // residual epilogue
    float *x;
    bf16 *xb;
    const bf16 *g_next;
    float *ss_out;
    // SwiGLU epilogue
    bf16 *h_out;
    // LM-head epilogue
    unsigned long long *keys;
    float *logits;
    int *argmax_out, *done_counter;
    int vocab;
};

template <int N>
struct GemmShape {
    static constexpr int BM = 128, BK = 64;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = N * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_RAW = (110 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int TMEM_COLS = N < 32 ? 32 : N;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
    static constexpr uint32_t IDESC = idesc_bf16(128, N);
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
};

constexpr int kGemmThreads = 192;

// ------------------------------------------------------------------ epilogues
// Each epilogue thread owns one output feature (TMEM lane) and sees 32 rows at
// a time (TMEM columns c0..c0+31) in v[].

struct EpiSmem {
    float rstd[160];
    float red[4][32];
    uint32_t am_val[4][32];
    uint32_t am_idx[4][32];
    int last;
};

__device__ __forceinline__ void epi_qkv(const GemmArgs &a, EpiSmem &es, float *xch, int tile, int c0, int R,
                                        float (&v)[32]) {
    const int f = threadIdx.x, warp = f >> 5, lane = f & 31;
    const int D = a.D, half = D >> 1;
    int section, head;  // 0 = q, 1 = k, 2 = v
    if (tile < a.q_tiles) {
        section = 0;
        head = (tile * 128 + f) / D;
    } else if (tile < a.q_tiles + a.k_tiles) {
        section = 1;
        head = ((tile - a.q_tiles) * 128 + f) / D;
    } else {
        section = 2;
        head = ((tile - a.q_tiles - a.k_tiles) * 128 + f) / D;
    }
    const int d = f % D;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= es.rstd[min(c0 + j, 159)];
    if (section < 2) {
        if (a.qk_norm) {
            float sq[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) sq[j] = v[j] * v[j];
            es.red[warp][lane] = transpose_sum32(sq, lane);
            named_bar_sync(1, 128);
            const int wph = D >> 5;               // warps per head
            const int w0 = (warp / wph) * wph;
            const float g = __bfloat162float(section == 0 ? a.q_gain[d] : a.k_gain[d]);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                float s = 0.f;
                for (int w = w0; w < w0 + wph; ++w) s += es.red[w][j];
                v[j] *= rsqrtf(s / static_cast<float>(D) + a.eps) * g;
            }
            named_bar_sync(1, 128);
        }
        // rotate-half RoPE: pair (d, d + D/2)
#pragma unroll
        for (int j = 0; j < 32; ++j) xch[j * 128 + f] = v[j];
        named_bar_sync(1, 128);
        const int partner = d < half ? f + half : f - half;
        const int jj = d < half ? d : d - half;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = c0 + j;
            if (r < R) {
                int pos = a.row_pos[r];
                pos = pos < 0 ? 0 : (pos >= a.rope_rows ? a.rope_rows - 1 : pos);
                const float2 cs = a.rope[static_cast<size_t>(pos) * half + jj];
                const float u = xch[j * 128 + partner];
                v[j] = d < half ? v[j] * cs.x - u * cs.y : v[j] * cs.x + u * cs.y;
            }
        }
        named_bar_sync(1, 128);
    }
    if (section == 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = c0 + j;
            if (r < R) a.q_out[(static_cast<size_t>(r) * a.nq + head) * D + d] = __float2bfloat16(v[j]);
        }
    } else {
        const int kvsel = section - 1;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int r = c0 + j;
            if (r < R) {
                const int seq = a.row_seq[r], pos = a.row_pos[r];
                const int slot_idx = pos / a.page_size;
                int page = -1;
                if (seq >= 0 && pos >= 0 && slot_idx < a.pages_per_seq)
                    page = a.page_table[static_cast<size_t>(seq) * a.pages_per_seq + slot_idx];
                if (page < 0 || page >= a.n_pages) {
                    set_status(a.status, SDV_ERR_CAPACITY);
                } else {
                    const size_t off =
                        ((((static_cast<size_t>(page) * 2 + kvsel) * a.nkv + head) * a.page_size + pos % a.page_size) *
                         D) +
                        d;
                    a.kv_layer[off] = __float2bfloat16(v[j]);
                }
            }
        }
    }
}

__device__ __forceinline__ void epi_resid(const GemmArgs &a, EpiSmem &es, int tile, int c0, int R, float (&v)[32]) {
    const int f = threadIdx.x, warp = f >> 5, lane = f & 31;
    const int F = tile * 128 + f;
    const bool valid = F < a.n_out;
    const float g = valid ? __bfloat162float(a.g_next[F]) : 0.f;
    float sq[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const int r = c0 + j;
        sq[j] = 0.f;
        if (valid && r < R) {
            const size_t o = static_cast<size_t>(r) * a.hidden + F;
            const float xn = a.x[o] + v[j];
            a.x[o] = xn;
            a.xb[o] = __float2bfloat16(xn * g);
            sq[j] = xn * xn;
        }
    }
    es.red[warp][lane] = transpose_sum32(sq, lane);
    named_bar_sync(1, 128);
    if (f < 32 && c0 + f < R)
        a.ss_out[static_cast<size_t>(tile) * a.rows_cap + c0 + f] =
            (es.red[0][f] + es.red[1][f]) + (es.red[2][f] + es.red[3][f]);
    named_bar_sync(1, 128);
}

__device__ __forceinline__ void epi_swiglu(const GemmArgs &a, EpiSmem &es, float *xch, int tile, int c0, int R,
                                           float (&v)[32]) {
    const int f = threadIdx.x, warp = f >> 5;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= es.rstd[min(c0 + j, 159)];
    if (warp >= 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) xch[j * 64 + (f - 64)] = v[j];
    }
    named_bar_sync(1, 128);
    if (warp < 2) {
        const int F = tile * 64 + f;
        if (F < a.n_out) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = c0 + j;
                if (r < R) {
                    const float gt = v[j], up = xch[j * 64 + f];
                    const float act = gt / (1.f + __expf(-gt));
                    a.h_out[static_cast<size_t>(r) * a.n_out + F] = __float2bfloat16(act * up);
                }
            }
        }
    }
    named_bar_sync(1, 128);
}

__device__ __forceinline__ void epi_lmhead(const GemmArgs &a, EpiSmem &es, int tile, int c0, int R, float (&v)[32]) {
    const int f = threadIdx.x, warp = f >> 5, lane = f & 31;
    const int vi = tile * 128 + f;
    const bool valid = vi < a.vocab;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= es.rstd[min(c0 + j, 159)];
    if (a.logits != nullptr && valid) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j < R) a.logits[static_cast<size_t>(c0 + j) * a.vocab + vi] = v[j];
    }
    uint32_t my_val = 0, my_idx = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const uint32_t u = valid ? orderable(v[j]) : 0u;
        const uint32_t m = __reduce_max_sync(0xffffffffu, u);
        const uint32_t cand = (valid && u == m) ? static_cast<uint32_t>(vi) : 0xffffffffu;
        const uint32_t idx = __reduce_min_sync(0xffffffffu, cand);
        if (lane == j) {
            my_val = m;
            my_idx = idx;
        }
    }
    es.am_val[warp][lane] = my_val;
    es.am_idx[warp][lane] = my_idx;
    named_bar_sync(1, 128);
    if (f < 32 && c0 + f < R) {
        uint32_t bv = es.am_val[0][f], bi = es.am_idx[0][f];
#pragma unroll
        for (int w = 1; w < 4; ++w) {
            const uint32_t cv = es.am_val[w][f], ci = es.am_idx[w][f];
            if (cv > bv || (cv == bv && ci < bi)) {
                bv = cv;
                bi = ci;
            }
        }
        atomicMax(&a.keys[c0 + f], (static_cast<unsigned long long>(bv) << 32) | (0xffffffffull - bi));
    }
    named_bar_sync(1, 128);
}

template <int KIND>
__device__ __forceinline__ void epi_dispatch(const GemmArgs &a, EpiSmem &es, float *xch, int tile, int c0, int R,
                                             float (&v)[32]) {
    if constexpr (KIND == EPI_QKV) epi_qkv(a, es, xch, tile, c0, R, v);
    else if constexpr (KIND == EPI_RESID) epi_resid(a, es, tile, c0, R, v);
    else if constexpr (KIND == EPI_SWIGLU) epi_swiglu(a, es, xch, tile, c0, R, v);
    else epi_lmhead(a, es, tile, c0, R, v);
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

template <int N, int KIND>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    using S = GemmShape<N>;
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

    // partial tile for the cluster reduction: [N rows][128 features] fp32 at the start
    // of the stage memory; exchange buffers for the epilogues after it.
    float *red = reinterpret_cast<float *>(smem);
    float *xch = reinterpret_cast<float *>(smem + N * 512);

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
            pdl_wait();  // activations come from the previous kernel
            for (int i = 0; i < pre; ++i)
                tma_load_2d(smem + i * S::STAGE_BYTES + S::A_BYTES, &tmB, &full_bar[i], (kb0 + i) * 64, 0);
            for (int i = pre; i < nk; ++i) {
                const int s = i % S::STAGES;
                const uint32_t ph = (i / S::STAGES) & 1;
                if (!mbar_wait(&empty_bar[s], ph ^ 1)) {
                    set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[s], S::STAGE_BYTES);
                uint8_t *sa = smem + s * S::STAGE_BYTES;
                const int kc = (kb0 + i) * 64;
                load_a<KIND>(sa, &tmA0, &tmA1, &tmA2, &full_bar[s], a, tile, kc, pol_w);
                tma_load_2d(sa + S::A_BYTES, &tmB, &full_bar[s], kc, 0);
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
                const uint64_t ad = sw128_desc(smem_u32(smem + s * S::STAGE_BYTES));
                const uint64_t bd = sw128_desc(smem_u32(smem + s * S::STAGE_BYTES + S::A_BYTES));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_bf16(tmem, ad + 2 * k, bd + 2 * k, S::IDESC, (i > 0 || k > 0) ? 1u : 0u);
                umma_commit(&empty_bar[s]);
            }
            umma_commit(&accum_bar);
        }
    }

    int R = 0;
    if (warp < 4) {
        // ---------------- epilogue warps 0-3: rstd rows, then the accumulator
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
        named_bar_sync(1, 128);
        if (!mbar_wait(&accum_bar, 0)) set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float v[32];
        if (clustered) {
            const int f = threadIdx.x;
            for (int c0 = 0; c0 < R; c0 += 32) {
                tmem_ld32(taddr + c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < R) red[(c0 + j) * 128 + f] = v[j];
            }
        } else {
            for (int c0 = 0; c0 < R; c0 += 32) {
                tmem_ld32(taddr + c0, v);
                epi_dispatch<KIND>(a, es, xch, tile, c0, R, v);
            }
        }
    }
    if (clustered) {
        // every partial of the tile is parked in its CTA's shared memory
        cluster_sync();
        if (warp < 4) {
            const int f = threadIdx.x;
            const int per = (R + a.splits - 1) / a.splits;
            const int s0 = min(R, static_cast<int>(cluster_ctarank()) * per), s1 = min(R, s0 + per);
            const uint32_t red_local = smem_u32(red);
            float v[32];
            for (int c0 = s0; c0 < s1; c0 += 32) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
                for (int q = 0; q < a.splits; ++q) {  // fixed split order
                    const uint32_t base = mapa_shared(red_local, static_cast<uint32_t>(q));
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < s1) v[j] += ld_dsmem(base + static_cast<uint32_t>(((c0 + j) * 128 + f) * 4));
                }
                epi_dispatch<KIND>(a, es, xch, tile, c0, s1, v);
            }
        }
        // no CTA leaves while its partial may still be read
        cluster_sync();
    }
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
}

}  // namespace sdv
