// Paged GQA attention for the verify span. K/V arrive by TMA: the pool is a 5-D tensor
// [layer*page][K|V][kv head][slot][dim], and one 128-key chunk of a kv head is, per page, a box of
// (page size) rows x 64 dims per half of the head dimension, landing 128-byte swizzled.
//
// A (sequence, 1024-position key group, kv head) is served by `splits` CTAs, each owning
// 8 / splits consecutive 128-key chunks of the group (the split is fixed per context, so a row's
// arithmetic never depends on the span). A CTA walks its chunks in position order with the next
// chunk's K/V copy in flight while the current chunk is computed (two shared-memory buffers), and
// keeps an online softmax (running max m, sum l, unnormalised o) per query row. At most 32 query
// rows (heads x span rows) per launch; warp w handles query tile w & 1 against the fixed 32-key
// quarter w >> 1 of every chunk (all eight warps busy at verify widths); the four quarters merge in
// shared memory at the end, in quarter order. When one CTA covers the whole key range it writes the
// output; otherwise every CTA parks its partial and the last to arrive merges all partials in
// position order, staging them in shared memory a block of rows at a time.
//
// Keys are cut by position only and a chunk that is fully masked for a row leaves that row's
// state exactly unchanged (scale 1, nothing added), so a row's result does not depend on how many
// span rows share the launch. Query rows and probabilities enter the tensor cores as bf16 hi/lo
// pairs; the output is written as a hi/lo pair.
#pragma once

#include "attention.cuh"

namespace sdv {

constexpr int kGrpThreads = 256;
constexpr int kGrpChunks = kAttnGroup / kAttnChunk;  // 8 chunks of 128 keys
constexpr int kGrpRows = 32;                         // query rows (heads x span rows) per launch
constexpr int kGrpQuarters = 4;                      // fixed key partition of a chunk
constexpr int kGrpQKeys = kAttnChunk / kGrpQuarters;

template <int D>
struct GrpShape {
    static constexpr int ROW = D * 2;
    static constexpr int Q_BYTES = 2 * kGrpRows * ROW;       // hi rows 0..31, lo rows 32..63
    static constexpr int HALF = kAttnChunk * 128;            // one 64-dim half of a chunk's K (or V)
    static constexpr int KV_BYTES = kAttnChunk * ROW;        // K (or V) of one chunk: D / 64 halves
    static constexpr int NBUF = 3;                           // chunks in flight + the one computed
    static constexpr int BUF_OFF = Q_BYTES;                  // buffers: [NBUF][K | V]
    static constexpr int ML_OFF = Q_BYTES + NBUF * 2 * KV_BYTES;
    static constexpr int SMEM = ML_OFF + 2 * kAttnRows * 8 + 1024;  // + alignment slack
    // after the loop the buffer region holds the four key quarters' fp32 partials [32][D]
    static_assert(NBUF * 2 * KV_BYTES >= kGrpQuarters * kGrpRows * D * 4, "partials must fit in the buffer region");
    static_assert(2 * kAttnRows * 8 >= kGrpQuarters * kGrpRows * 8, "quarter statistics must fit");
};

// byte offset of 16-byte piece c of key row r in a K or V chunk buffer: 64-dim halves of 128
// keys x 128 bytes each, 128-byte swizzled (the TMA layout)
__device__ __forceinline__ uint32_t swz_kv(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (kAttnChunk * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kGrpThreads, 1)
    attn_group_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tkv) {
    using S = GrpShape<D>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sm;
    __shared__ int page_s[kAttnGroup / 1 + 1];  // page of every position block of the group
    __shared__ int last_s;
    __shared__ __align__(8) uint64_t full[3];

    pdl_trigger();
    pdl_wait();
    // optional timeline: 0 start, 1 Q and page ids in, 2 first chunk landed, 3 chunks done, 4 quarters
    // merged, 5 partial parked, 6 parts merged, 7 end; merge: 8 statistics staged, 9 weights done
    auto stamp = [&](int ev) {
        if (a.trace && threadIdx.x == 0)
            a.trace[(static_cast<size_t>(blockIdx.y) * gridDim.x + blockIdx.x) * 16 + ev] = globaltimer();
    };
    stamp(0);
    const int w = blockIdx.x / a.splits, sp = blockIdx.x % a.splits, g = blockIdx.y;
    if (w >= *a.n_work) return;
    const int4 wi = a.work[w];
    const int b = wi.x & 0xffff, grp_idx = wi.x >> 16;
    const int L = wi.y, S_b = wi.z, row0 = wi.w;
    const int ni = max(0, min(S_b - a.q0, a.qrows));
    if (ni == 0) return;
    const int M = a.grp * ni, Mpad = (M + 15) & ~15;
    const int key_end = L + S_b;
    const int n_groups = (key_end + kAttnGroup - 1) / kAttnGroup;
    const int g0 = grp_idx * kAttnGroup, g1 = min(g0 + kAttnGroup, key_end);
    const int n_ch_group = (g1 - g0 + kAttnChunk - 1) / kAttnChunk;
    const int c_per = kGrpChunks / a.splits;
    const int c_lo = sp * c_per, c_hi = min(c_lo + c_per, n_ch_group);  // this CTA's chunks (may be none)
    const int n_ch = max(0, c_hi - c_lo);
    const int n_parts = n_groups * a.splits;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t head_stride = static_cast<size_t>(a.page_size) * D;
    const bool has_lo = a.q_plane != 0;

    // Q rows j = i_local * grp + hh (span row q0 + i_local, head g*grp + hh), both planes
    for (int e = tid; e < 2 * Mpad * CH; e += kGrpThreads) {
        const int pl = e / (Mpad * CH), j = (e / CH) % Mpad, c = e % CH;
        const bool valid = j < M && (pl == 0 || has_lo);
        const bf16 *src = a.q;
        if (valid) {
            const int r = row0 + a.q0 + j / a.grp;
            const int h = g * a.grp + j % a.grp;
            src = a.q + pl * a.q_plane + (static_cast<size_t>(r) * a.nq + h) * D + c * 8;
        }
        cp_async16(smem_u32(sQ) + swz<D>(pl * kGrpRows + j, c), src, valid);
    }
    cp_async_commit();
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&full[2], 1);
        fence_mbar_init();
        prefetch_tensormap(&tkv);
    }
    const int pg0 = g0 / a.page_size, npg = (g1 - 1) / a.page_size - pg0 + 1;
    for (int i = tid; i < npg; i += kGrpThreads) {
        const int slot_idx = pg0 + i;
        page_s[i] = slot_idx < a.pages_per_seq ? a.page_table[static_cast<size_t>(b) * a.pages_per_seq + slot_idx] : -1;
    }
    __syncthreads();

    // one chunk's K and V: per page of the chunk, per 64-dim half, one box (thread 0 issues)
    const int ppc = kAttnChunk / a.page_size;  // pages per chunk
    auto load_chunk = [&](int ch, int buf) {  // ch: this CTA's chunk index
        if (tid != 0) return;
        uint8_t *kb = sm + S::BUF_OFF + buf * 2 * S::KV_BYTES;
        const int k0 = g0 + (c_lo + ch) * kAttnChunk, k1 = min(k0 + kAttnChunk, g1);
        const int p_first = k0 / a.page_size - pg0, p_last = (k1 - 1) / a.page_size - pg0;
        int bytes = 0;
        for (int pi = p_first; pi <= p_last; ++pi) {
            const int page = page_s[pi];
            if (page >= 0 && page < a.n_pages) bytes += 2 * (D / 64) * a.page_size * 128;
        }
        mbar_arrive_expect_tx(&full[buf], static_cast<uint32_t>(bytes));
        for (int pi = p_first; pi <= p_last; ++pi) {
            const int page = page_s[pi];
            if (page < 0 || page >= a.n_pages) {
                set_status(a.status, SDV_ERR_CAPACITY);
                continue;
            }
            const int row = (pi - p_first) * a.page_size;
            const int e = a.layer * a.n_pages + page;
#pragma unroll
            for (int kv = 0; kv < 2; ++kv)
#pragma unroll
                for (int h = 0; h < D / 64; ++h)
                    tma_load_5d(kb + kv * S::KV_BYTES + h * S::HALF + row * 128, &tkv, &full[buf], h * 64, 0, g, kv, e);
        }
    };
    __syncthreads();  // barriers initialised, page ids in place
    if (n_ch > 0) load_chunk(0, 0);
    if (n_ch > 1) load_chunk(1, 1);
    if (n_ch > 2) load_chunk(2, 2);
    cp_async_wait_all();  // Q
    __syncthreads();
    stamp(1);
    (void)ppc;

    // warp w: query tile mt = w & 1 (16 of the <= 32 rows), 32-key quarter kq = w >> 1 of every chunk
    const int mt = warp & 1, kq = warp >> 1;
    const bool active = mt * 16 < M;
    const int gq = lane >> 2, tq = lane & 3;
    const int jr0 = mt * 16 + gq, jr1 = jr0 + 8;
    const int lim0 = L + a.q0 + jr0 / a.grp, lim1 = L + a.q0 + jr1 / a.grp;
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int ch = 0; ch < n_ch; ++ch) {
        const int buf = ch % S::NBUF;
        if (!mbar_wait(&full[buf], (ch / S::NBUF) & 1)) set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
        if (ch == 0) stamp(2);
        const uint32_t sK = smem_u32(sm + S::BUF_OFF + buf * 2 * S::KV_BYTES), sV = sK + S::KV_BYTES;
        {   // keys past the group end read as zero V rows (the pool holds stale data there)
            const int kstart = g0 + (c_lo + ch) * kAttnChunk, nvalid = min(kAttnChunk, g1 - kstart);
            for (int e = tid; e < (kAttnChunk - nvalid) * CH; e += kGrpThreads) {
                const int r = nvalid + e / CH, c = e % CH;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sV + swz_kv(r, c)), "r"(0u) : "memory");
            }
        }
        __syncthreads();
        const int ubase = g0 + (c_lo + ch) * kAttnChunk + kq * kGrpQKeys;
        if (active && ubase < g1) {
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll 2
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t qh[4], ql[4];
                {
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int c = ks * 2 + (lane >> 4);
                    ldsm_x4(smem_u32(sQ) + swz<D>(row, c), qh[0], qh[1], qh[2], qh[3]);
                    if (has_lo) ldsm_x4(smem_u32(sQ) + swz<D>(kGrpRows + row, c), ql[0], ql[1], ql[2], ql[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 4; nt += 2) {
                    const int i = lane >> 3;
                    const int key = kq * kGrpQKeys + nt * 8 + (i >> 1) * 8 + (lane & 7);
                    const int c = ks * 2 + (i & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(sK + swz_kv(key, c), b0, b1, b2, b3);
                    mma_bf16_16816(s[nt], qh, b0, b1);
                    mma_bf16_16816(s[nt + 1], qh, b2, b3);
                    if (has_lo) {
                        mma_bf16_16816(s[nt], ql, b0, b1);
                        mma_bf16_16816(s[nt + 1], ql, b2, b3);
                    }
                }
            }
            // mask (position < group end and <= the row's causal limit), running max (log2 domain)
            float mx0 = m0, mx1 = m1;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int u = ubase + nt * 8 + tq * 2 + e;
                    const bool ok0 = u < g1 && u <= lim0, ok1 = u < g1 && u <= lim1;
                    s[nt][e] = ok0 ? s[nt][e] * a.scale_log2 : -INFINITY;
                    s[nt][2 + e] = ok1 ? s[nt][2 + e] * a.scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, s[nt][e]);
                    mx1 = fmaxf(mx1, s[nt][2 + e]);
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            // rescale the running state to the new max (exactly 1 when the max did not move)
            const float sc0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mx0), sc1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mx1);
            m0 = mx0;
            m1 = mx1;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                o[dn][0] *= sc0;
                o[dn][1] *= sc0;
                o[dn][2] *= sc1;
                o[dn][3] *= sc1;
            }
            const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
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
                for (int dn = 0; dn < D / 8; dn += 2) {
                    const int i = lane >> 3;
                    const int key = kq * kGrpQKeys + kk * 16 + (i & 1) * 8 + (lane & 7);
                    const int c = dn + (i >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(sV + swz_kv(key, c), b0, b1, b2, b3);
                    mma_bf16_16816(o[dn], ph, b0, b1);
                    mma_bf16_16816(o[dn + 1], ph, b2, b3);
                    if (a.p_lo) {
                        mma_bf16_16816(o[dn], pl, b0, b1);
                        mma_bf16_16816(o[dn + 1], pl, b2, b3);
                    }
                }
            }
            rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
            rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
            rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
            rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
            l0 = l0 * sc0 + rs0;
            l1 = l1 * sc1 + rs1;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic accesses before the refill
        __syncthreads();  // buffer `buf` is free
        if (ch + S::NBUF < n_ch) load_chunk(ch + S::NBUF, buf);
    }

    stamp(3);
    // the four quarters' states -> shared memory [quarter][row][D] (rows without keys stay (-inf, 0, 0)),
    // merged per row in quarter order into quarter 0's slots
    float *qo = reinterpret_cast<float *>(sm + S::BUF_OFF);
    float2 *qml = reinterpret_cast<float2 *>(sm + S::ML_OFF);  // [quarter][kGrpRows]
    if (mt * 16 < Mpad) {
        float *dst = qo + static_cast<size_t>(kq) * kGrpRows * D;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            *reinterpret_cast<float2 *>(&dst[jr0 * D + dn * 8 + tq * 2]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(&dst[jr1 * D + dn * 8 + tq * 2]) = make_float2(o[dn][2], o[dn][3]);
        }
        if (tq == 0) {
            qml[kq * kGrpRows + jr0] = make_float2(m0, l0);
            qml[kq * kGrpRows + jr1] = make_float2(m1, l1);
        }
    }
    __syncthreads();
    __shared__ float qw_s[kGrpRows][kGrpQuarters];
    __shared__ float2 mlf_s[kGrpRows];
    for (int j = tid; j < Mpad; j += kGrpThreads) {  // per row: merged (m, l) and the quarters' weights
        float Mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kGrpQuarters; ++q) Mx = fmaxf(Mx, qml[q * kGrpRows + j].x);
        float l = 0.f;
#pragma unroll
        for (int q = 0; q < kGrpQuarters; ++q) {
            const float2 ml = qml[q * kGrpRows + j];
            const float wq = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
            qw_s[j][q] = wq;
            l += wq * ml.y;
        }
        mlf_s[j] = make_float2(Mx, l);
    }
    __syncthreads();
    for (int e4 = tid; e4 < Mpad * D / 4; e4 += kGrpThreads) {
        const int j = e4 / (D / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kGrpQuarters; ++q) {
            const float wq = qw_s[j][q];
            const float4 x = reinterpret_cast<const float4 *>(qo + static_cast<size_t>(q) * kGrpRows * D)[e4];
            acc.x += wq * x.x;
            acc.y += wq * x.y;
            acc.z += wq * x.z;
            acc.w += wq * x.w;
        }
        reinterpret_cast<float4 *>(qo)[e4] = acc;
    }
    __syncthreads();
    stamp(4);
    float *po_s = qo;  // [row][D] unnormalised o of this CTA's keys
    float2 *ml_s = mlf_s;

    auto store = [&](int j, int d, float v) {
        const int r = row0 + a.q0 + j / a.grp, h = g * a.grp + j % a.grp;
        const size_t oi = (static_cast<size_t>(r) * a.nq + h) * D + d;
        const Bf16Pair pr = split_bf16(v);
        a.out[oi] = pr.hi;
        if (a.out_plane) a.out[oi + a.out_plane] = pr.lo;
    };
    if (n_parts == 1) {
        for (int e = tid; e < M * D; e += kGrpThreads) store(e / D, e % D, po_s[e] / ml_s[e / D].y);
        stamp(7);
        return;
    }
    // park this CTA's partial; the last of (b, g) to arrive merges every part in position order
    const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
    const size_t slot = (static_cast<size_t>(w) * a.splits + sp) * a.nkv + g;
    for (int e = tid; e < M * D; e += kGrpThreads) a.part_o[(slot * rowsw + e / D) * D + e % D] = po_s[e];
    for (int j = tid; j < M; j += kGrpThreads) a.part_ml[slot * rowsw + j] = ml_s[j];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int *cnt = &a.counters[(b * a.nkv + g) * kAttnCluster];
        const int last = atomicAdd(cnt, 1) == n_parts - 1;
        if (last) *cnt = 0;
        last_s = last;
    }
    __syncthreads();
    stamp(5);
    if (!last_s) return;
    __threadfence();
    // parts of (b, g) in position order: part p = (group wfirst + p / splits, split p % splits); the
    // work items of one sequence are consecutive
    const int wfirst = w - grp_idx;
    auto part_slot = [&](int p) {
        return (static_cast<size_t>(wfirst) * a.splits + p) * a.nkv + g;
    };
    // (m, l) of every part and row, staged; per row the max Mx, each part's weight exp2(m - Mx) and
    // the denominator; then each thread owns four-column groups of the output and adds the parts'
    // o in part order from registers, loads for a batch of parts in flight together
    if (n_parts * kGrpRows * 12 + kGrpRows * 4 > S::NBUF * 2 * S::KV_BYTES) {  // (over ~340 parts)
        if (tid == 0) set_status(a.status, SDV_ERR_UNSUPPORTED);
        return;
    }
    float2 *sml = reinterpret_cast<float2 *>(sm + S::BUF_OFF);          // [part][kGrpRows]
    float *swt = reinterpret_cast<float *>(sml + n_parts * kGrpRows);     // [part][kGrpRows]
    float *sden = swt + n_parts * kGrpRows;                               // [kGrpRows]
    for (int e = tid; e < n_parts * M; e += kGrpThreads) {
        const int p = e / M, j = e - p * M;
        sml[p * kGrpRows + j] = __ldcg(&a.part_ml[part_slot(p) * rowsw + j]);
    }
    __syncthreads();
    stamp(8);
    for (int j = tid; j < M; j += kGrpThreads) {
        float Mx = -INFINITY;
        for (int p = 0; p < n_parts; ++p) Mx = fmaxf(Mx, sml[p * kGrpRows + j].x);
        float den = 0.f;
        for (int p = 0; p < n_parts; ++p) {
            const float2 ml = sml[p * kGrpRows + j];
            const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
            swt[p * kGrpRows + j] = sc;
            den += sc * ml.y;
        }
        sden[j] = den;
    }
    __syncthreads();
    stamp(9);
    constexpr int PB = 4;                                   // parts per batch
    constexpr int PER = kGrpRows * (D / 4) / kGrpThreads;   // four-column groups per thread
    float4 num[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) num[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < n_parts; p0 += PB) {
        float4 x[PER][PB];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e4 = tid + i * kGrpThreads, j = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
#pragma unroll
            for (int k = 0; k < PB; ++k)
                if (j < M && p0 + k < n_parts)
                    x[i][k] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (part_slot(p0 + k) * rowsw + j) * D + d));
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = (tid + i * kGrpThreads) / (D / 4);
#pragma unroll
            for (int k = 0; k < PB; ++k)
                if (j < M && p0 + k < n_parts) {
                    const float sc = swt[(p0 + k) * kGrpRows + j];
                    num[i].x += sc * x[i][k].x;
                    num[i].y += sc * x[i][k].y;
                    num[i].z += sc * x[i][k].z;
                    num[i].w += sc * x[i][k].w;
                }
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e4 = tid + i * kGrpThreads, j = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
        if (j >= M) continue;
        const float den = sden[j];
        store(j, d, num[i].x / den);
        store(j, d + 1, num[i].y / den);
        store(j, d + 2, num[i].z / den);
        store(j, d + 3, num[i].w / den);
    }
    stamp(6);
}

}  // namespace sdv
