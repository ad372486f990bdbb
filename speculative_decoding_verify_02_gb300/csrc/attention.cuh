// Paged grouped-query attention for the verify span.
//
// Query rows and probabilities enter the tensor cores as bf16 hi/lo pairs
// (two MMAs each), so only the stored K/V carry bf16 rounding; the output is
// written as a hi/lo pair for the O projection.
//
// Keys are cut by position only (never by span length): 128-key chunks, and
// groups of 8 chunks (1024 positions). A group of one sequence and one kv
// head is one work item, run by a thread-block cluster of 8 CTAs: CTA c loads
// chunk c of the group (its K/V pages, one shot) and the query rows of the kv
// head's q-head group (grp heads x span rows, one 16-row MMA tile per warp),
// and runs the softmax with the causal limit "row i attends positions <=
// L_b + i" (L_b is read from device memory at run time). The 8 chunk partials
// (m, l, o) are merged over distributed shared memory in chunk order. A
// sequence of one group writes its output there; longer sequences park one
// partial per group in global memory, and for each row slice the last group
// to arrive merges all groups in group order. Every row's reduction order is
// thus fixed by positions alone.
#pragma once

#include "common.cuh"

namespace sdv {

struct AttnArgs {
    const bf16 *q;           // [rows][nq][D] (hi plane), lo plane q_plane elements later
    size_t q_plane;          // 0: q has no lo plane
    const bf16 *kv_layer;    // pool + layer offset: [page][2][nkv][P][D]
    const int *page_table;   // [max_batch][pages_per_seq]
    int pages_per_seq, page_size, n_pages;
    const int4 *work;        // [n] (b | group << 16, L_b, S_b, first row of b)
    const int *n_work;       // [1]
    int nq, nkv, D, grp;
    int q0, qrows;           // span rows q0 .. q0+qrows-1 handled by this launch (grp*qrows <= 64)
    float scale_log2;        // log2(e) / sqrt(D)
    float *part_o;           // [work][nkv][grp*qrows][D]  group partials (unnormalised o)
    float2 *part_ml;         // [work][nkv][grp*qrows]     (m, l)
    int *counters;           // [max_batch][nkv][kAttnCluster] group arrivals per row slice
    bf16 *out;               // [rows][nq*D] (hi plane), lo plane out_plane elements later
    size_t out_plane;        // 0: write the hi plane only (a plain bf16 output)
    int *status;
    int splits;              // attention_group.cuh: CTAs sharing one group's chunks (1, 2, 4 or 8)
    int group;               // attention_group.cuh: key positions per group (1024 or 2048)
    int p_lo;                // attention_group.cuh: 1 = probabilities as a hi/lo pair, 0 = bf16 only
    int layer;               // attention_group.cuh: layer index in the pool tensor map
    int merge_groups;        // attention_group.cuh: sequences of up to this many key groups are merged
                             // inside the attention kernel; longer ones by attn_merge_kernel
    int window;              // attention_group.cuh: > 0 on a sliding-window layer (ring of `window` positions)
    int max_span;            // rows per sequence held by swa_backup
    const bf16 *swa_backup;  // the layer's copies of the ring slots the span overwrote [max_batch][max_span][K|V][nkv][D]
    unsigned long long *trace;  // attention_group.cuh: optional [CTA][8] %globaltimer stamps, or nullptr
};

constexpr int kAttnThreads = 256;   // 8 warps: 4 query tiles x 2 key blocks
constexpr int kAttnKB = 64;         // keys per MMA block
constexpr int kAttnChunk = 128;     // keys per CTA
constexpr int kAttnCluster = 8;     // CTAs (chunks) per work item
constexpr int kAttnGroup = kAttnChunk * kAttnCluster;
constexpr int kAttnRows = 64;       // query rows per launch (grp heads x span rows)

template <int D>
struct AttnShape {
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int Q_BYTES = 2 * kAttnRows * ROW_BYTES;        // hi and lo planes
    static constexpr int KV_BYTES = kAttnChunk * ROW_BYTES;          // K (or V) of one chunk
    static constexpr int SMEM = Q_BYTES + 2 * KV_BYTES + 2 * kAttnRows * 8;
    // after the softmax the K/V region holds two fp32 partials [64 rows][D] (one per key block)
    static_assert(2 * KV_BYTES >= 2 * kAttnRows * D * 4, "partials must fit in the K/V region");
};

// byte offset of 16-byte chunk `c` of row `r` in a row-major tile with an XOR swizzle
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * D * 2 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(bf16 lo, bf16 hi) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}
__device__ __forceinline__ float ld_dsmem_rank(const void *local, uint32_t rank) {
    return ld_dsmem(mapa_shared(smem_u32(local), rank));
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_kernel(const AttnArgs a) {
    using S = AttnShape<D>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t *sQ = sm;                                                          // hi rows 0..63, lo rows 64..127
    const uint32_t sK = smem_u32(sm + S::Q_BYTES);
    const uint32_t sV = smem_u32(sm + S::Q_BYTES + S::KV_BYTES);
    float *po_s = reinterpret_cast<float *>(sm + S::Q_BYTES);                 // after compute: [64][D]
    float *po2_s = po_s + kAttnRows * D;                                      // second key block's partial
    float2 *ml_s = reinterpret_cast<float2 *>(sm + S::Q_BYTES + 2 * S::KV_BYTES);
    float2 *ml2_s = ml_s + kAttnRows;
    __shared__ int last_s;
    __shared__ int page_s[kAttnChunk];  // page ids of the chunk's positions (at most one per key)

    pdl_trigger();
    pdl_wait();
    const int w = blockIdx.x / kAttnCluster, g = blockIdx.y;
    const int cr = static_cast<int>(cluster_ctarank());
    // Both early exits depend only on (w, b), which the 8 CTAs of a cluster share,
    // so a cluster leaves whole and never waits on a departed CTA.
    const int4 wi = a.work[w];  // (the list has room for every CTA's index; stale past n_work)
    if (w >= *a.n_work) return;
    const int b = wi.x & 0xffff, grp_idx = wi.x >> 16;
    const int L = wi.y, S_b = wi.z, row0 = wi.w;
    const int ni = max(0, min(S_b - a.q0, a.qrows));
    if (ni == 0) return;
    const int M = a.grp * ni;
    const int key_end = L + S_b;
    const int n_groups = (key_end + kAttnGroup - 1) / kAttnGroup;
    const int k0 = (grp_idx * kAttnCluster + cr) * kAttnChunk;
    const int k1 = min(k0 + kAttnChunk, key_end);
    const int nblk = k1 > k0 ? (k1 - k0 + kAttnKB - 1) / kAttnKB : 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t head_stride = static_cast<size_t>(a.page_size) * D;
    const int Mpad = (M + 15) & ~15;
    const bool has_lo = a.q_plane != 0;

    // stage Q rows j = i_local * grp + hh (span row q0 + i_local, head g*grp + hh), both planes,
    // and the chunk's K/V
    if (nblk > 0) {
        for (int e = tid; e < 2 * Mpad * CH; e += kAttnThreads) {
            const int pl = e / (Mpad * CH), j = (e / CH) % Mpad, ch = e % CH;
            const bool valid = j < M && (pl == 0 || has_lo);
            const bf16 *src = a.q;
            if (valid) {
                const int r = row0 + a.q0 + j / a.grp;
                const int h = g * a.grp + j % a.grp;
                src = a.q + pl * a.q_plane + (static_cast<size_t>(r) * a.nq + h) * D + ch * 8;
            }
            cp_async16(smem_u32(sQ) + swz<D>(pl * kAttnRows + j, ch), src, valid);
        }
        const int nkeys = nblk * kAttnKB;
        // page id of every page the chunk touches, looked up once
        const int pg0 = k0 / a.page_size, npg = (k1 - 1) / a.page_size - pg0 + 1;
        for (int i = tid; i < npg; i += kAttnThreads) {
            const int slot_idx = pg0 + i;
            page_s[i] = slot_idx < a.pages_per_seq ? a.page_table[b * a.pages_per_seq + slot_idx] : -1;
        }
        __syncthreads();
        for (int e = tid; e < nkeys * CH; e += kAttnThreads) {
            const int key = e / CH, ch = e % CH;
            const int u = k0 + key;
            bool valid = u < k1;
            const bf16 *srcK = a.kv_layer, *srcV = a.kv_layer;
            if (valid) {
                const int page = page_s[u / a.page_size - pg0];
                if (page < 0 || page >= a.n_pages) {
                    set_status(a.status, SDV_ERR_CAPACITY);
                    valid = false;
                } else {
                    const size_t base = (static_cast<size_t>(page) * 2 * a.nkv + g) * head_stride +
                                        static_cast<size_t>(u % a.page_size) * D + ch * 8;
                    srcK = a.kv_layer + base;
                    srcV = a.kv_layer + base + static_cast<size_t>(a.nkv) * head_stride;
                }
            }
            cp_async16(sK + swz<D>(key, ch), srcK, valid);
            cp_async16(sV + swz<D>(key, ch), srcV, valid);
        }
        cp_async_commit();
        cp_async_wait_all();
    }
    __syncthreads();

    const int mt = warp & 3, blk = warp >> 2;  // query tile, and which 64-key block of the chunk
    const bool active = blk < nblk && mt * 16 < M;
    const int gq = lane >> 2, tq = lane & 3;
    const int jr0 = mt * 16 + gq, jr1 = jr0 + 8;
    const int lim0 = L + a.q0 + jr0 / a.grp, lim1 = L + a.q0 + jr1 / a.grp;

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
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
                const int ch = ks * 2 + (lane >> 4);
                ldsm_x4(smem_u32(sQ) + swz<D>(row, ch), qh[0], qh[1], qh[2], qh[3]);
                ldsm_x4(smem_u32(sQ) + swz<D>(kAttnRows + row, ch), ql[0], ql[1], ql[2], ql[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 8; nt += 2) {
                const int i = lane >> 3;
                const int key = blk * kAttnKB + nt * 8 + (i >> 1) * 8 + (lane & 7);
                const int ch = ks * 2 + (i & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sK + swz<D>(key, ch), b0, b1, b2, b3);
                mma_bf16_16816(s[nt], qh, b0, b1);
                mma_bf16_16816(s[nt + 1], qh, b2, b3);
                if (has_lo) {
                    mma_bf16_16816(s[nt], ql, b0, b1);
                    mma_bf16_16816(s[nt + 1], ql, b2, b3);
                }
            }
        }
        // mask and softmax of the block (log2 domain)
        const int ubase = k0 + blk * kAttnKB;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int u = ubase + nt * 8 + tq * 2 + e;
                const bool ok0 = u < k1 && u <= lim0, ok1 = u < k1 && u <= lim1;
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
        m0 = mx0;
        m1 = mx1;
        const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
        float rs0 = 0.f, rs1 = 0.f;
        // P = exp2(s - m) one 16-key step at a time, as a hi/lo pair: the A operand of P.V
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
            for (int dn = 0; dn < D / 8; dn += 2) {
                const int i = lane >> 3;
                const int key = blk * kAttnKB + kk * 16 + (i & 1) * 8 + (lane & 7);
                const int ch = dn + (i >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sV + swz<D>(key, ch), b0, b1, b2, b3);
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
    __syncthreads();  // K/V no longer read: the region now holds the two key blocks' partials

    // key-block partials -> shared memory ([row][D] fp32 and (m, l)); rows without keys stay (-inf, 0, 0)
    if (mt * 16 < Mpad) {
        float *dst = blk == 0 ? po_s : po2_s;
        float2 *mld = blk == 0 ? ml_s : ml2_s;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
            *reinterpret_cast<float2 *>(&dst[jr0 * D + dn * 8 + tq * 2]) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(&dst[jr1 * D + dn * 8 + tq * 2]) = make_float2(o[dn][2], o[dn][3]);
        }
        if (tq == 0) {
            mld[jr0] = make_float2(m0, l0);
            mld[jr1] = make_float2(m1, l1);
        }
    }
    __syncthreads();
    // the chunk's partial: block 0 merged with block 1
    for (int e = tid; e < Mpad * D; e += kAttnThreads) {
        const int j = e / D;
        const float2 A = ml_s[j], Bp = ml2_s[j];
        const float Mx = fmaxf(A.x, Bp.x);
        const float sa = A.x == -INFINITY ? 0.f : exp2f(A.x - Mx), sb = Bp.x == -INFINITY ? 0.f : exp2f(Bp.x - Mx);
        po_s[e] = po_s[e] * sa + po2_s[e] * sb;
    }
    __syncthreads();
    for (int j = tid; j < Mpad; j += kAttnThreads) {
        const float2 A = ml_s[j], Bp = ml2_s[j];
        const float Mx = fmaxf(A.x, Bp.x);
        const float sa = A.x == -INFINITY ? 0.f : exp2f(A.x - Mx), sb = Bp.x == -INFINITY ? 0.f : exp2f(Bp.x - Mx);
        ml_s[j] = make_float2(Mx, A.y * sa + Bp.y * sb);
    }
    cluster_sync();

    // merge the 8 chunks of the group for this CTA's row slice, chunk order 0..7
    const int per = (M + kAttnCluster - 1) / kAttnCluster;
    const int r0 = min(M, cr * per), r1 = min(M, r0 + per);
    const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
    const size_t slot = static_cast<size_t>(w) * a.nkv + g;
    for (int e = tid; e < (r1 - r0) * D; e += kAttnThreads) {
        const int j = r0 + e / D, d = e % D;
        float mq[kAttnCluster];
        float Mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < kAttnCluster; ++q) {
            mq[q] = ld_dsmem_rank(&ml_s[j].x, static_cast<uint32_t>(q));
            Mx = fmaxf(Mx, mq[q]);
        }
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int q = 0; q < kAttnCluster; ++q) {
            const float sc = mq[q] == -INFINITY ? 0.f : exp2f(mq[q] - Mx);
            den += sc * ld_dsmem_rank(&ml_s[j].y, static_cast<uint32_t>(q));
            num += sc * ld_dsmem_rank(&po_s[j * D + d], static_cast<uint32_t>(q));
        }
        const int r = row0 + a.q0 + j / a.grp;
        const int h = g * a.grp + j % a.grp;
        if (n_groups == 1) {
            const size_t oi = (static_cast<size_t>(r) * a.nq + h) * D + d;
            const Bf16Pair pr = split_bf16(num / den);
            a.out[oi] = pr.hi;
            if (a.out_plane) a.out[oi + a.out_plane] = pr.lo;
        } else {
            a.part_o[(slot * rowsw + j) * D + d] = num;
            if (d == 0) a.part_ml[slot * rowsw + j] = make_float2(Mx, den);
        }
    }
    cluster_sync();  // no CTA leaves while its partial may still be read

    if (n_groups > 1) {
        // the last group to finish this row slice merges every group, in group order
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int *cnt = &a.counters[(b * a.nkv + g) * kAttnCluster + cr];
            last_s = atomicAdd(cnt, 1) == n_groups - 1;
            if (last_s) *cnt = 0;
        }
        __syncthreads();
        if (last_s) {
            __threadfence();
            const int wfirst = w - grp_idx;  // the work items of one sequence are consecutive
            for (int e = tid; e < (r1 - r0) * D; e += kAttnThreads) {
                const int j = r0 + e / D, d = e % D;
                float Mx = -INFINITY;
                for (int gi = 0; gi < n_groups; ++gi) {
                    const size_t sl = (static_cast<size_t>(wfirst + gi) * a.nkv + g) * rowsw + j;
                    Mx = fmaxf(Mx, __ldcg(&a.part_ml[sl].x));
                }
                float num = 0.f, den = 0.f;
                for (int gi = 0; gi < n_groups; ++gi) {
                    const size_t sl = (static_cast<size_t>(wfirst + gi) * a.nkv + g) * rowsw + j;
                    const float2 ml = __ldcg(&a.part_ml[sl]);
                    const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - Mx);
                    den += sc * ml.y;
                    num += sc * __ldcg(&a.part_o[sl * D + d]);
                }
                const int r = row0 + a.q0 + j / a.grp;
                const int h = g * a.grp + j % a.grp;
                const size_t oi = (static_cast<size_t>(r) * a.nq + h) * D + d;
                const Bf16Pair pr = split_bf16(num / den);
                a.out[oi] = pr.hi;
                if (a.out_plane) a.out[oi + a.out_plane] = pr.lo;
            }
        }
    }
}

}  // namespace sdv
