// Paged grouped-query attention for the verify span.
//
// Each sequence's keys 0 .. L_b+S_b-1 are cut into fixed chunks of positions
// (the cut depends on positions only, never on the span length). One CTA takes
// one (sequence, chunk, kv head): it stages the query rows of the kv head's
// q-head group (grp heads x span rows, one 16-row MMA tile per warp) and
// streams the chunk's K/V pages in 64-key blocks, running an online softmax
// with the causal limit "row i attends positions <= L_b + i". The KV length
// is read from device memory at run time. A second kernel merges the chunk
// partials (m, l, o) in chunk order with a log-sum-exp rescale.
#pragma once

#include "common.cuh"

namespace sdv {

struct AttnArgs {
    const bf16 *q;           // [rows][nq][D]
    const bf16 *kv_layer;    // pool + layer offset: [page][2][nkv][P][D]
    const int *page_table;   // [max_batch][pages_per_seq]
    int pages_per_seq, page_size, n_pages;
    const int *seq_base;     // [B] cache length before the span
    const int *row_off;      // [B+1]
    const int *work;         // [n] (b << 16) | chunk
    const int *work_off;     // [B+1] first work item of each sequence
    const int *n_work;       // [1]
    const int *row_seq;      // [rows] sequence of each packed row
    const int *nrows;        // [1]
    int nq, nkv, D, grp;
    int chunk;               // keys per work item (multiple of 64)
    int q0, qrows;           // span rows q0 .. q0+qrows-1 handled by this launch
    float scale_log2;        // log2(e) / sqrt(D)
    float *part_o;           // [work][nkv][grp*qrows][D]
    float2 *part_ml;         // [work][nkv][grp*qrows]
    bf16 *out;               // [rows][nq*D]
    int *status;
};

constexpr int kAttnThreads = 256;  // 8 warps, one 16-row query tile each
constexpr int kAttnKB = 64;        // keys per streamed block

template <int D>
struct AttnShape {
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int Q_BYTES = 128 * ROW_BYTES;
    static constexpr int KV_BYTES = kAttnKB * ROW_BYTES;            // one of K or V, one block
    static constexpr int SMEM = Q_BYTES + 4 * KV_BYTES + 128;       // Q + double-buffered K and V
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
template <int n>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(n) : "memory");
}

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
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_partial_kernel(const AttnArgs a) {
    using S = AttnShape<D>;
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t sm[];
    uint8_t *sQ = sm;
    const uint32_t sK0 = smem_u32(sm + S::Q_BYTES);                 // K buffers 0/1, then V buffers 0/1
    const uint32_t sV0 = smem_u32(sm + S::Q_BYTES + 2 * S::KV_BYTES);

    pdl_trigger();
    pdl_wait();
    const int w = blockIdx.x, g = blockIdx.y;
    if (w >= *a.n_work) return;
    const int b = a.work[w] >> 16, c = a.work[w] & 0xffff;
    const int L = a.seq_base[b];
    const int S_b = a.row_off[b + 1] - a.row_off[b];
    const int ni = min(S_b - a.q0, a.qrows);
    if (ni <= 0) return;
    const int M = a.grp * ni;
    const int key_end = L + S_b;
    const int k0 = c * a.chunk;
    const int k1 = min(k0 + a.chunk, key_end);
    const int nblk = (k1 - k0 + kAttnKB - 1) / kAttnKB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t head_stride = static_cast<size_t>(a.page_size) * D;

    // stage Q rows j = i_local * grp + hh (row i = q0 + i_local of the span, head g*grp + hh)
    for (int e = tid; e < 128 * CH; e += kAttnThreads) {
        const int j = e / CH, ch = e % CH;
        const bool valid = j < M;
        const bf16 *src = a.q;
        if (valid) {
            const int r = a.row_off[b] + a.q0 + j / a.grp;
            const int h = g * a.grp + j % a.grp;
            src = a.q + (static_cast<size_t>(r) * a.nq + h) * D + ch * 8;
        }
        cp_async16(smem_u32(sQ) + swz<D>(j, ch), src, valid);
    }
    auto load_kv = [&](int blk, int buf) {
        for (int e = tid; e < kAttnKB * CH; e += kAttnThreads) {
            const int key = e / CH, ch = e % CH;
            const int u = k0 + blk * kAttnKB + key;
            bool valid = u < k1;
            const bf16 *srcK = a.kv_layer, *srcV = a.kv_layer;
            if (valid) {
                const int slot_idx = u / a.page_size;
                const int page = slot_idx < a.pages_per_seq ? a.page_table[b * a.pages_per_seq + slot_idx] : -1;
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
            cp_async16(sK0 + buf * S::KV_BYTES + swz<D>(key, ch), srcK, valid);
            cp_async16(sV0 + buf * S::KV_BYTES + swz<D>(key, ch), srcV, valid);
        }
        cp_async_commit();
    };
    load_kv(0, 0);  // commit group 0 holds Q and the first K/V block

    const int mt = warp;                  // 16-row query tile of this warp
    const bool active = mt * 16 < M;
    const int gq = lane >> 2, tq = lane & 3;
    // causal limits of this thread's two rows (gq and gq + 8 of the tile)
    const int jr0 = mt * 16 + gq, jr1 = jr0 + 8;
    const int lim0 = L + a.q0 + jr0 / a.grp, lim1 = L + a.q0 + jr1 / a.grp;

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int blk = 0; blk < nblk; ++blk) {
        const int buf = blk & 1;
        if (blk + 1 < nblk) {
            load_kv(blk + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (active) {
            // scores for 64 keys: 8 n-tiles of 8 keys
            float s[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t qa[4];
                {
                    const int row = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = ks * 2 + (lane >> 4);
                    ldsm_x4(smem_u32(sQ) + swz<D>(row, ch), qa[0], qa[1], qa[2], qa[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 8; nt += 2) {
                    const int i = lane >> 3;
                    const int key = nt * 8 + (i >> 1) * 8 + (lane & 7);
                    const int ch = ks * 2 + (i & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(sK0 + buf * S::KV_BYTES + swz<D>(key, ch), b0, b1, b2, b3);
                    mma_bf16_16816(s[nt], qa, b0, b1);
                    mma_bf16_16816(s[nt + 1], qa, b2, b3);
                }
            }
            // mask and online softmax (log2 domain)
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
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
            m0 = mn0;
            m1 = mn1;
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn) {
                o[dn][0] *= al0;
                o[dn][1] *= al0;
                o[dn][2] *= al1;
                o[dn][3] *= al1;
            }
            // P = exp2(s - m) one 16-key step at a time, consumed at once as the A operand of P.V
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t pa[4];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int nt = 2 * kk + hf;
                    const float p0 = exp2f(s[nt][0] - base0), p1 = exp2f(s[nt][1] - base0);
                    const float p2 = exp2f(s[nt][2] - base1), p3 = exp2f(s[nt][3] - base1);
                    rs0 += p0 + p1;
                    rs1 += p2 + p3;
                    pa[2 * hf] = pack_bf16(p0, p1);
                    pa[2 * hf + 1] = pack_bf16(p2, p3);
                }
#pragma unroll
                for (int dn = 0; dn < D / 8; dn += 2) {
                    const int i = lane >> 3;
                    const int key = kk * 16 + (i & 1) * 8 + (lane & 7);
                    const int ch = dn + (i >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(sV0 + buf * S::KV_BYTES + swz<D>(key, ch), b0, b1, b2, b3);
                    mma_bf16_16816(o[dn], pa, b0, b1);
                    mma_bf16_16816(o[dn + 1], pa, b2, b3);
                }
            }
            rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
            rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
            rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
            rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
        }
        __syncthreads();  // the buffer is refilled next iteration
    }

    if (active) {
        const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
        const size_t slot = static_cast<size_t>(w) * a.nkv + g;  // one partial per (work item, kv head)
        float *po = a.part_o + slot * rowsw * D;
        float2 *pml = a.part_ml + slot * rowsw;
        if (jr0 < M) {
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn)
                *reinterpret_cast<float2 *>(&po[static_cast<size_t>(jr0) * D + dn * 8 + tq * 2]) =
                    make_float2(o[dn][0], o[dn][1]);
            if (tq == 0) pml[jr0] = make_float2(m0, l0);
        }
        if (jr1 < M) {
#pragma unroll
            for (int dn = 0; dn < D / 8; ++dn)
                *reinterpret_cast<float2 *>(&po[static_cast<size_t>(jr1) * D + dn * 8 + tq * 2]) =
                    make_float2(o[dn][2], o[dn][3]);
            if (tq == 0) pml[jr1] = make_float2(m1, l1);
        }
    }
}

// One CTA per (packed row, kv head); thread d of the block handles dim d of each head in the group.
__global__ void attn_combine_kernel(const AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, g = blockIdx.y, d = threadIdx.x;
    if (r >= *a.nrows) return;
    const int b = a.row_seq[r];
    const int i = r - a.row_off[b];
    if (i < a.q0 || i >= a.q0 + a.qrows) return;
    const int w0 = a.work_off[b], w1 = a.work_off[b + 1];
    const size_t rowsw = static_cast<size_t>(a.grp) * a.qrows;
    for (int hh = 0; hh < a.grp; ++hh) {
        const int j = (i - a.q0) * a.grp + hh;
        float M = -INFINITY;
        for (int w = w0; w < w1; ++w) M = fmaxf(M, a.part_ml[(w * a.nkv + g) * rowsw + j].x);
        float num = 0.f, den = 0.f;
        for (int w = w0; w < w1; ++w) {
            const size_t slot = (static_cast<size_t>(w) * a.nkv + g) * rowsw + j;
            const float2 ml = a.part_ml[slot];
            const float sc = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            den += sc * ml.y;
            num += sc * a.part_o[slot * a.D + d];
        }
        a.out[static_cast<size_t>(r) * a.nq * a.D + (g * a.grp + hh) * a.D + d] = __float2bfloat16(num / den);
    }
}

}  // namespace sdv
