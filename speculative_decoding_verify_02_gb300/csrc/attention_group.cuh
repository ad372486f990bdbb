// Paged GQA attention for the verify span. K/V arrive by TMA: the pool is a 5-D tensor
// [layer*page][K|V][kv head][slot][dim], and one 128-key chunk of a kv head is, per page, a box of
// (page size) rows x 64 dims per half of the head dimension, landing 128-byte swizzled.
//
// A (sequence, key group, kv head) is served by one thread-block cluster of `splits` CTAs, each
// owning group / 128 / splits consecutive 128-key chunks of the group; the group (1024 positions,
// or 2048 where that brings a long sequence's grid into one wave) and the split are fixed per
// configuration, so a row's arithmetic never depends on the span or the batch. In each CTA one
// producer warp issues the chunks' K/V copies into a ring of three buffers, refilling a buffer as
// soon as every consumer warp released it, and eight consumer warps walk the chunks in position
// order keeping an online softmax (running max m, sum l, unnormalised o) per query row. At most 32
// query rows (heads x span rows) per launch; consumer warp w handles query tile w & 1 against the
// fixed 32-key quarter w >> 1 of every chunk. The quarter states stay in shared memory; after a
// cluster barrier each CTA merges a slice of the rows over all splits x 4 states of the group,
// reading the other CTAs' shared memory, in position order. With one key group that is the output;
// with several, each group's state is parked in global memory and merged across the groups, in
// group order: when a group's cluster has at least four CTAs, sequences of up to 8 groups by the
// last group CTA of each split index to finish (a few rows each); every other multi-group
// sequence by attn_merge_kernel, with one CTA per four rows.
//
// Keys are cut by position only and a chunk that is fully masked for a row leaves that row's
// state exactly unchanged (scale 1, nothing added), so a row's result does not depend on how many
// span rows share the launch. Query rows and probabilities enter the tensor cores as bf16 hi/lo
// pairs; the output is written as a hi/lo pair.
#pragma once

#include "attention.cuh"

namespace sdv {

constexpr int kGrpConsumers = 256;                  // 8 warps: query tile x key quarter
constexpr int kGrpThreads = kGrpConsumers + 32;      // + 1 producer warp that issues the K/V copies
constexpr int kMaxKvHeads = 16;
// the KV pool's tensor maps, one per kv head (kernel parameter space)
struct KvMaps {
    CUtensorMap m[kMaxKvHeads];
};
constexpr int kGrpMaxSplits = kAttnCluster;         // CTAs of a group's cluster: 1, 2, 4 or 8
constexpr int kGrpRows = 32;                         // query rows (heads x span rows) per launch
constexpr int kGrpQuarters = 4;                      // fixed key partition of a chunk
constexpr int kGrpQKeys = kAttnChunk / kGrpQuarters;
// sequences of up to this many key groups are merged across groups inside the
// attention kernel (by the last group CTA to finish); longer ones by attn_merge_kernel
constexpr int kInKernelMergeGroups = 8;

template <int D>
struct GrpShape {
    static constexpr int ROW = D * 2;
    static constexpr int Q_BYTES = 2 * kGrpRows * ROW;       // hi rows 0..31, lo rows 32..63
    static constexpr int KV_BYTES = kAttnChunk * ROW;        // K (or V) of one chunk: D / 64 halves
    static constexpr int NBUF = 3;                           // chunks in flight + the one computed
    static constexpr int BUF_OFF = Q_BYTES;                  // buffers: [NBUF][K | V]
    static constexpr int ML_OFF = Q_BYTES + NBUF * 2 * KV_BYTES;
    static constexpr int SMEM = ML_OFF + 2 * kAttnRows * 8 + 1024;  // + alignment slack
    // after the loop the buffer region holds the four key quarters' fp32 partials [32][D]
    // quarter states after the loop: fp32 rows of D + 8 (the stride keeps a warp's float2 stores of
    // eight rows x four column pairs on distinct banks)
    static constexpr int QO_LD = D + 8;
    // quarter states [quarter][32 rows][QO_LD], then the CTA's merged state [32 rows][QO_LD]
    static constexpr int RECV_OFF = kGrpQuarters * kGrpRows * QO_LD * 4;
    static_assert(NBUF * 2 * KV_BYTES >= RECV_OFF + kGrpRows * QO_LD * 4, "states must fit in the buffer region");
    static_assert(2 * kAttnRows * 8 >= kGrpQuarters * kGrpRows * 8, "quarter statistics must fit");
};

// A chunk buffer holds, per page of the chunk, the page's K box then its V box; a box is lines
// (half * P + slot) of 128 bytes, 128-byte swizzled (the TMA layout). Byte offset of 16-byte piece
// c of key r (kv = 0 K, 1 V), for page size P = 1 << lp (P >= 8) and head dimension D.
template <int D>
__device__ __forceinline__ uint32_t swz_kv(int r, int c, int kv, int lp) {
    const int P = 1 << lp;
    return static_cast<uint32_t>(((r >> lp) * 2 + kv) * (P * D * 2) + ((c >> 3) * P + (r & (P - 1))) * 128 +
                                 (((c & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kGrpThreads, 1)
    attn_group_kernel(const AttnArgs a, const __grid_constant__ KvMaps tkv) {
    using S = GrpShape<D>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = sm;
    __shared__ __align__(8) uint64_t full[S::NBUF], empty[S::NBUF];
    __shared__ int last_s;

    pdl_trigger();
    // The forward's prepare kernel finished before this kernel started (it does not trigger its
    // dependents early), so the work list, the page table and the K/V of every position before the
    // span (written by earlier steps) are final here: they are read, and the copies of chunks that
    // hold only such positions issued, before the wait. The span's own K/V and the queries come
    // from the QKV projection this kernel follows, after the wait.
    // optional timeline: 0 start, 1 Q in, 2 first chunk landed, 3 chunks done, 4 the CTA states of
    // the cluster in place, 5 cluster merge done (output or parked group state), 6 CTA end; 10 second
    // chunk landed, 11 second chunk computed, 12 last chunk landed (when there are more than two);
    // the CTA merging across key groups: 13 merge started, 14 group weights staged, 15 first
    // element summed, 8 merge done
    auto stamp = [&](int ev) {
        if (a.trace && threadIdx.x == 0)
            a.trace[((static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * 16 + ev] =
                globaltimer();
    };
    // grid (splits, kv heads, work items): the CTAs of one wave cover every kv head, so their K/V
    // reads spread over whole pages of the pool
    const int w = blockIdx.z, sp = blockIdx.x, g = blockIdx.y;
    const int n_work = *a.n_work;
    const int4 wi = a.work[w];  // w < work_cap: inside the list (both loads in flight together)
    if (w >= n_work) return;    // the whole cluster shares w, so it leaves together
    const int b = wi.x & 0xffff, grp_idx = wi.x >> 16;
    const int L = wi.y, S_b = wi.z, row0 = wi.w;
    const int ni = max(0, min(S_b - a.q0, a.qrows));
    if (ni == 0) return;
    const int M = a.grp * ni, Mpad = (M + 15) & ~15;
    const int key_end = L + S_b;
    const int n_groups = (key_end + a.group - 1) / a.group;
    const int g0 = grp_idx * a.group, g1 = min(g0 + a.group, key_end);
    const int n_ch_group = (g1 - g0 + kAttnChunk - 1) / kAttnChunk;
    const int c_per = a.group / kAttnChunk / a.splits;
    // this CTA's chunks (may be none); on a sliding-window layer the chunks below every span row's
    // window are skipped (all their keys are masked, so they would leave the state unchanged)
    const int win_lo = a.window > 0 ? max(0, L - a.window + 1) : 0;
    const int c_lo = max(sp * c_per, a.window > 0 ? (win_lo - g0) / kAttnChunk : 0);
    const int c_hi = min(sp * c_per + c_per, n_ch_group);
    const int n_ch = max(0, c_hi - c_lo);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool consumer = tid < kGrpConsumers;
    const bool has_lo = a.q_plane != 0;
    const int lp = 31 - __clz(a.page_size);  // page size: a power of two in [8, 128]

    if (tid == 0) {
        for (int i = 0; i < S::NBUF; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGrpConsumers / 32);  // one arrival per consumer warp
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (!consumer) {
        // Producer warp: one chunk's K and V is one box per page of the chunk (K and V rows of head
        // g, both 64-dim halves, 8 KB at page size 16), issued by the lanes after lane 0 has
        // posted the byte count; a buffer is refilled once every consumer warp released it. The
        // page ids come straight from the page table, so the first copies start while Q loads.
        prefetch_tensormap(&tkv.m[g]);
        const uint64_t pol_kv = policy_evict_first();  // K/V are read once per step: keep L2 for the rest
        const int box_bytes = 2 * a.page_size * D * 2;
        // leading chunks of positions before the span only (not on a sliding-window layer, whose
        // ring slots the QKV projection overwrites): issued before the wait
        int pre = 0;
        while (a.window == 0 && pre < min(n_ch, S::NBUF) &&
               min(g0 + (c_lo + pre + 1) * kAttnChunk, g1) <= L)
            ++pre;
        bool waited = false;
        for (int ch = 0; ch < n_ch; ++ch) {
            const int buf = ch % S::NBUF;
            if (ch == pre) {
                pdl_wait();
                waited = true;
            }
            if (ch >= S::NBUF && !mbar_wait(&empty[buf], ((ch / S::NBUF) - 1) & 1)) {
                if (lane == 0) set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
                break;
            }
            uint8_t *kb = sm + S::BUF_OFF + buf * 2 * S::KV_BYTES;
            const int k0 = g0 + (c_lo + ch) * kAttnChunk, k1 = min(k0 + kAttnChunk, g1);
            const int s_first = k0 / a.page_size, s_last = (k1 - 1) / a.page_size;  // page-table slots
            int page = -1;
            const int si = s_first + lane;
            // a sliding-window layer's positions live in a ring over the first window / page_size slots
            const int ts = a.window > 0 ? si % (a.window / a.page_size) : si;
            if (si <= s_last && ts < a.pages_per_seq) page = a.page_table[static_cast<size_t>(b) * a.pages_per_seq + ts];
            const bool ok = page >= 0 && page < a.n_pages;
            if (si <= s_last && !ok) set_status(a.status, SDV_ERR_CAPACITY);
            const int bytes = __reduce_add_sync(0xffffffffu, ok ? box_bytes : 0);
            if (lane == 0) mbar_arrive_expect_tx(&full[buf], static_cast<uint32_t>(bytes));
            __syncwarp();
            if (ok)
                tma_load_5d_hint(kb + (si - s_first) * box_bytes, &tkv.m[g], &full[buf], 0, 0, 0, 0,
                                 a.layer * a.n_pages + page, pol_kv);
        }
        if (!waited) pdl_wait();
    } else {
        pdl_wait();
        stamp(0);
        // Q rows j = i_local * grp + hh (span row q0 + i_local, head g*grp + hh), both planes
        for (int e = tid; e < 2 * Mpad * CH; e += kGrpConsumers) {
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
        cp_async_wait_all();
        named_bar_sync(1, kGrpConsumers);  // Q in place for every consumer warp
        stamp(1);
    }

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

    for (int ch = 0; consumer && ch < n_ch; ++ch) {
        const int buf = ch % S::NBUF;
        if (!mbar_wait(&full[buf], (ch / S::NBUF) & 1)) set_status(a.status, SDV_ERR_DEVICE_TIMEOUT);
        if (ch == 0) stamp(2);
        if (ch == 1) stamp(10);
        if (ch == n_ch - 1 && ch > 1) stamp(12);
        const uint32_t sKV = smem_u32(sm + S::BUF_OFF + buf * 2 * S::KV_BYTES);
        {   // keys past the group end read as zero V rows (the pool holds stale data there)
            const int kstart = g0 + (c_lo + ch) * kAttnChunk, nvalid = min(kAttnChunk, g1 - kstart);
            // sliding-window layer: the span rows overwrote the ring slots of positions
            // L - window .. L + S_b - 1 - window; those still in a row's window are read from the
            // layer's backup instead (span row j kept position L + j - window)
            const int ev_lo = max(kstart, max(win_lo, L - a.window)), ev_hi = min(kstart + nvalid, L + S_b - a.window);
            const int n_ev = a.window > 0 ? max(0, ev_hi - ev_lo) : 0;
            if (nvalid < kAttnChunk || n_ev > 0) {  // the same for every consumer warp
                for (int e = tid; e < (kAttnChunk - nvalid) * CH; e += kGrpConsumers) {
                    const int r = nvalid + e / CH, c = e % CH;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sKV + swz_kv<D>(r, c, 1, lp)), "r"(0u) : "memory");
                }
                for (int e = tid; e < n_ev * 2 * CH; e += kGrpConsumers) {
                    const int u = ev_lo + e / (2 * CH), kv = (e / CH) & 1, c = e % CH;
                    const int j = u - (L - a.window);
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        a.swa_backup + ((static_cast<size_t>(b) * a.max_span + j) * 2 + kv) * a.nkv * D + g * D + c * 8);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(sKV + swz_kv<D>(u - kstart, c, kv, lp)),
                                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                named_bar_sync(1, kGrpConsumers);
            }
        }
        const int ubase = g0 + (c_lo + ch) * kAttnChunk + kq * kGrpQKeys;
        if (active && ubase < g1) {
            float s[4][4], t[4][4];  // q_hi . k and q_lo . k, summed after the k loop
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = t[nt][0] = t[nt][1] = t[nt][2] = t[nt][3] = 0.f;
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
                    ldsm_x4(sKV + swz_kv<D>(key, c, 0, lp), b0, b1, b2, b3);
                    mma_bf16_16816(s[nt], qh, b0, b1);
                    mma_bf16_16816(s[nt + 1], qh, b2, b3);
                    if (has_lo) {
                        mma_bf16_16816(t[nt], ql, b0, b1);
                        mma_bf16_16816(t[nt + 1], ql, b2, b3);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                s[nt][0] += t[nt][0];
                s[nt][1] += t[nt][1];
                s[nt][2] += t[nt][2];
                s[nt][3] += t[nt][3];
            }
            // mask (position < group end and <= the row's causal limit), running max (log2 domain)
            float mx0 = m0, mx1 = m1;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int u = ubase + nt * 8 + tq * 2 + e;
                    bool ok0 = u < g1 && u <= lim0, ok1 = u < g1 && u <= lim1;
                    if (a.window > 0) {  // sliding window: the row's last `window` positions
                        ok0 = ok0 && u > lim0 - a.window;
                        ok1 = ok1 && u > lim1 - a.window;
                    }
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
                    ldsm_x4_t(sKV + swz_kv<D>(key, c, 1, lp), b0, b1, b2, b3);
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
        if (ch == 1) stamp(11);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic accesses before the refill
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[buf])) : "memory");
    }
    // every chunk consumed by every consumer warp (no copy in flight) before the buffers are reused
    __syncthreads();

    stamp(3);
    // the four quarters' states -> shared memory: per [quarter][row] a row of QO_LD floats holding
    // the unnormalised o, then (m, l) at D, D + 1; quarters without keys keep (-inf, 0, 0)
    float *qo = reinterpret_cast<float *>(sm + S::BUF_OFF);
    if (consumer && mt * 16 < Mpad) {
        float *dst = qo + static_cast<size_t>(kq) * kGrpRows * S::QO_LD;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            *reinterpret_cast<float2 *>(&dst[jr0 * S::QO_LD + dn * 8 + tq * 2]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(&dst[jr1 * S::QO_LD + dn * 8 + tq * 2]) = make_float2(o[dn][2], o[dn][3]);
        }
        if (tq == 0) {
            *reinterpret_cast<float2 *>(&dst[jr0 * S::QO_LD + D]) = make_float2(m0, l0);
            *reinterpret_cast<float2 *>(&dst[jr1 * S::QO_LD + D]) = make_float2(m1, l1);
        }
    }
    __syncthreads();
    auto store = [&](int j, int d, float v) {
        const int r = row0 + a.q0 + j / a.grp, h = g * a.grp + j % a.grp;
        const size_t oi = (static_cast<size_t>(r) * a.nq + h) * D + d;
        const Bf16Pair pr = split_bf16(v);
        a.out[oi] = pr.hi;
        if (a.out_plane) a.out[oi + a.out_plane] = pr.lo;
    };
    const bool multi = n_groups > 1;
    const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
    const size_t gslot = static_cast<size_t>(w) * a.nkv + g;  // this group's parked state (multi)
    if (a.splits == 1) {
        // One CTA per group: merging its quarters gives the group's state directly, the output of
        // a single-group sequence or the state parked for the merge across groups (the same values
        // the cluster merge below gives with one split, whose weight is exactly 1).
        for (int e = tid; e < M * (D / 4); e += kGrpThreads) {
            const int j = e / (D / 4), d = (e % (D / 4)) * 4;
            float2 st[kGrpQuarters];
            float Mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kGrpQuarters; ++k) {
                st[k] = *reinterpret_cast<const float2 *>(&qo[(k * kGrpRows + j) * S::QO_LD + D]);
                Mx = fmaxf(Mx, st[k].x);
            }
            float wq[kGrpQuarters];
#pragma unroll
            for (int k = 0; k < kGrpQuarters; ++k) wq[k] = st[k].x == -INFINITY ? 0.f : exp2f(st[k].x - Mx);
            float l = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kGrpQuarters; ++k) {
                l += wq[k] * st[k].y;
                const float4 x = *reinterpret_cast<const float4 *>(&qo[(k * kGrpRows + j) * S::QO_LD + d]);
                acc.x += wq[k] * x.x;
                acc.y += wq[k] * x.y;
                acc.z += wq[k] * x.z;
                acc.w += wq[k] * x.w;
            }
            if (!multi) {
                store(j, d, acc.x / l);
                store(j, d + 1, acc.y / l);
                store(j, d + 2, acc.z / l);
                store(j, d + 3, acc.w / l);
            } else {
                *reinterpret_cast<float4 *>(&a.part_o[(gslot * rowsw + j) * D + d]) = acc;
                if (d == 0) a.part_ml[gslot * rowsw + j] = make_float2(Mx, l);
            }
        }
        stamp(4);
        stamp(5);
        stamp(6);
        return;  // sequences of several groups are merged by attn_merge_kernel
    }
    // the CTA's state: quarters merged per row in quarter order -> cs [row][QO_LD] (o, then m, l)
    float *cs = qo + S::RECV_OFF / 4;
    for (int e = tid; e < M * (D / 4 + 1); e += kGrpThreads) {
        const int j = e / (D / 4 + 1), c4 = e % (D / 4 + 1);
        float2 st[kGrpQuarters];
        float Mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kGrpQuarters; ++k) {
            st[k] = *reinterpret_cast<const float2 *>(&qo[(k * kGrpRows + j) * S::QO_LD + D]);
            Mx = fmaxf(Mx, st[k].x);
        }
        float wq[kGrpQuarters];
#pragma unroll
        for (int k = 0; k < kGrpQuarters; ++k) wq[k] = st[k].x == -INFINITY ? 0.f : exp2f(st[k].x - Mx);
        if (c4 == D / 4) {  // the row's (m, l)
            float l = 0.f;
#pragma unroll
            for (int k = 0; k < kGrpQuarters; ++k) l += wq[k] * st[k].y;
            *reinterpret_cast<float2 *>(&cs[j * S::QO_LD + D]) = make_float2(Mx, l);
        } else {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kGrpQuarters; ++k) {
                const float4 x = *reinterpret_cast<const float4 *>(&qo[(k * kGrpRows + j) * S::QO_LD + c4 * 4]);
                acc.x += wq[k] * x.x;
                acc.y += wq[k] * x.y;
                acc.z += wq[k] * x.z;
                acc.w += wq[k] * x.w;
            }
            *reinterpret_cast<float4 *>(&cs[j * S::QO_LD + c4 * 4]) = acc;
        }
    }
    cluster_sync();  // every CTA's state of the group in place
    stamp(4);

    // Cluster merge: CTA `sp` finishes rows [j0, j1) over the splits' states, in split (position)
    // order, reading the other CTAs' shared memory. With one key group that is the output;
    // otherwise the group's (o, m, l) is parked for the merge across groups.
    const int per = (M + a.splits - 1) / a.splits;
    const int j0 = min(M, sp * per), j1 = min(M, j0 + per);
    const uint32_t cs_l = smem_u32(cs);
    for (int it = tid; it < (j1 - j0) * (D / 4); it += kGrpThreads) {
        const int j = j0 + it / (D / 4), d = (it % (D / 4)) * 4;
        float2 ml[kGrpMaxSplits];
        float4 x[kGrpMaxSplits];
        float Mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kGrpMaxSplits; ++c) {
            if (c < a.splits) {
                const uint32_t row = mapa_shared(cs_l, static_cast<uint32_t>(c)) + j * S::QO_LD * 4;
                ml[c] = ld_dsmem_f2(row + D * 4);
                x[c] = ld_dsmem_f4(row + d * 4);
                Mx = fmaxf(Mx, ml[c].x);
            }
        }
        float den = 0.f;
        float4 n = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kGrpMaxSplits; ++c) {
            if (c < a.splits) {
                const float wq = ml[c].x == -INFINITY ? 0.f : exp2f(ml[c].x - Mx);
                den += wq * ml[c].y;
                n.x += wq * x[c].x;
                n.y += wq * x[c].y;
                n.z += wq * x[c].z;
                n.w += wq * x[c].w;
            }
        }
        if (!multi) {
            store(j, d, n.x / den);
            store(j, d + 1, n.y / den);
            store(j, d + 2, n.z / den);
            store(j, d + 3, n.w / den);
        } else {
            *reinterpret_cast<float4 *>(&a.part_o[(gslot * rowsw + j) * D + d]) = n;
            if (d == 0) a.part_ml[gslot * rowsw + j] = make_float2(Mx, den);
        }
    }
    cluster_arrive();  // this CTA's reads of the other CTAs' shared memory are done
    stamp(5);
    if (multi && n_groups <= a.merge_groups) {
        // up to a.merge_groups (<= kInKernelMergeGroups) groups: the last of the groups' CTAs with
        // this split index merges rows [j0, j1) over the groups' parked states, in group order
        // (other sequences are merged by attn_merge_kernel)
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int *cnt = &a.counters[(b * a.nkv + g) * kAttnCluster + sp];
            const int last = atomicAdd(cnt, 1) == n_groups - 1;
            if (last) *cnt = 0;
            last_s = last;
        }
        __syncthreads();
        if (last_s) {
            __threadfence();
            stamp(13);
            const int wfirst = w - grp_idx;  // the work items of one sequence are consecutive
            const int nr = j1 - j0;
            auto slot_of = [&](int q) { return (static_cast<size_t>(wfirst) + q) * a.nkv + g; };
            // per row: the maximum over the groups, each group's weight and the denominator, staged
            // in shared memory (the quarter-state region, no longer read)
            float *gw = qo;                                            // [group][nr]
            float *gden = gw + kInKernelMergeGroups * kGrpRows;        // [nr]
            for (int r = tid; r < nr; r += kGrpThreads) {
                float2 st[kInKernelMergeGroups];
                float Mx = -INFINITY;
#pragma unroll
                for (int q = 0; q < kInKernelMergeGroups; ++q)
                    if (q < n_groups) {
                        st[q] = __ldcg(&a.part_ml[slot_of(q) * rowsw + j0 + r]);
                        Mx = fmaxf(Mx, st[q].x);
                    }
                float den = 0.f;
#pragma unroll
                for (int q = 0; q < kInKernelMergeGroups; ++q)
                    if (q < n_groups) {
                        const float wq = st[q].x == -INFINITY ? 0.f : exp2f(st[q].x - Mx);
                        gw[q * nr + r] = wq;
                        den += wq * st[q].y;
                    }
                gden[r] = den;
            }
            __syncthreads();
            stamp(14);
            // two float4 columns per thread and pass, every group's load in flight together
            for (int it0 = tid; it0 < nr * (D / 4); it0 += 2 * kGrpThreads) {
                float4 x[2][kInKernelMergeGroups];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int it = it0 + u * kGrpThreads;
                    const int j = j0 + it / (D / 4), d = (it % (D / 4)) * 4;
#pragma unroll
                    for (int q = 0; q < kInKernelMergeGroups; ++q)
                        if (it < nr * (D / 4) && q < n_groups)
                            x[u][q] = __ldcg(reinterpret_cast<const float4 *>(&a.part_o[(slot_of(q) * rowsw + j) * D + d]));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int it = it0 + u * kGrpThreads;
                    if (it >= nr * (D / 4)) break;
                    const int r = it / (D / 4), j = j0 + r, d = (it % (D / 4)) * 4;
                    float4 n = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int q = 0; q < kInKernelMergeGroups; ++q) {
                        if (q < n_groups) {  // group order
                            const float wq = gw[q * nr + r];
                            n.x += wq * x[u][q].x;
                            n.y += wq * x[u][q].y;
                            n.z += wq * x[u][q].z;
                            n.w += wq * x[u][q].w;
                        }
                    }
                    if (it == 0) stamp(15);
                    const float den = gden[r];
                    store(j, d, n.x / den);
                    store(j, d + 1, n.y / den);
                    store(j, d + 2, n.z / den);
                    store(j, d + 3, n.w / den);
                }
            }
            stamp(8);
        }
    }
    cluster_wait();  // no CTA leaves while another may still read its shared memory
    stamp(6);
}

// Merge across key groups (sequences of more than kInKernelMergeGroups groups): each group's state
// (unnormalised o, running max m, sum l) was parked by its cluster; CTA (slice, kv head g,
// sequence b) finishes kMergeRows query rows: per row the maximum over the groups, each group's
// weight 2^(m_q - max) (0 for a group with no key at or before the row), and the weighted sums of
// l and o in group order. Shorter sequences were finished by the attention kernel itself.
constexpr int kMergeRows = 4;

template <int D>
__global__ void __launch_bounds__(kMergeRows * D / 4)
    attn_merge_kernel(const AttnArgs a, const int *work_off) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.z, g = blockIdx.y;
    const int w0 = work_off[b], n_groups = work_off[b + 1] - w0;
    if (n_groups <= 1 || n_groups <= a.merge_groups) return;  // one group, or merged in the attention kernel
    const int4 wi = a.work[w0];
    const int S_b = wi.z, row0 = wi.w;
    const int ni = max(0, min(S_b - a.q0, a.qrows));
    const int M = a.grp * ni;
    const int j = blockIdx.x * kMergeRows + static_cast<int>(threadIdx.x) / (D / 4);
    const int d = (static_cast<int>(threadIdx.x) % (D / 4)) * 4;
    if (j >= M) return;
    const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
    auto slot = [&](int q) { return ((static_cast<size_t>(w0) + q) * a.nkv + g) * rowsw + j; };
    constexpr int QB = 8;  // groups whose loads are in flight together
    float Mx = -INFINITY;
    for (int q0 = 0; q0 < n_groups; q0 += QB) {
        float mx[QB];
#pragma unroll
        for (int k = 0; k < QB; ++k) mx[k] = q0 + k < n_groups ? __ldcg(&a.part_ml[slot(q0 + k)]).x : -INFINITY;
#pragma unroll
        for (int k = 0; k < QB; ++k) Mx = fmaxf(Mx, mx[k]);
    }
    float den = 0.f;
    float4 n = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < n_groups; q0 += QB) {
        float2 ml[QB];
        float4 x[QB];
#pragma unroll
        for (int k = 0; k < QB; ++k) {
            if (q0 + k < n_groups) {
                ml[k] = __ldcg(&a.part_ml[slot(q0 + k)]);
                x[k] = __ldcg(reinterpret_cast<const float4 *>(&a.part_o[slot(q0 + k) * D + d]));
            }
        }
#pragma unroll
        for (int k = 0; k < QB; ++k) {
            if (q0 + k < n_groups) {  // group order
                const float wq = ml[k].x == -INFINITY ? 0.f : exp2f(ml[k].x - Mx);
                den += wq * ml[k].y;
                n.x += wq * x[k].x;
                n.y += wq * x[k].y;
                n.z += wq * x[k].z;
                n.w += wq * x[k].w;
            }
        }
    }
    const int r = row0 + a.q0 + j / a.grp, h = g * a.grp + j % a.grp;
    const size_t oi = (static_cast<size_t>(r) * a.nq + h) * D + d;
    const float v[4] = {n.x / den, n.y / den, n.z / den, n.w / den};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const Bf16Pair pr = split_bf16(v[i]);
        a.out[oi + i] = pr.hi;
        if (a.out_plane) a.out[oi + i + a.out_plane] = pr.lo;
    }
}

}  // namespace sdv
