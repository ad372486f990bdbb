// Paged attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or an allocating framework routine):
// code that runs while a CUDA graph is being captured, plug-in interfaces that
// receive only the buffers of their inputs and outputs, and deployments whose
// device memory is fixed at start-up. This entry point runs the same paged
// attention kernel as sdv_op_attention without a context or workspace: its
// scratch (the attention work list, the per-slice group counters and the
// per-group partials of sequences longer than 1024 positions) lives in the
// file-scope array below, which every GPU that loads the library holds until
// the process exits.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "attention.cuh"
#include "common.cuh"

namespace {

using namespace sdv;

constexpr size_t kScratchBytes = 8u << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceSetup {
    bool done = false;
    unsigned char *scratch = nullptr;  // device address of g_scratch on that device
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mu;

// Scratch layout: [status int][n_work int][work list][counters][group partials (m, l)][group partials o]
struct Layout {
    size_t work, counters, ml, o, total;
};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

Layout layout(int B, int nkv, int D, int rows_per_item, int max_work) {
    Layout L;
    size_t off = 256;
    L.work = off;
    off = up256(off + sizeof(int4) * static_cast<size_t>(max_work));
    L.counters = off;
    off = up256(off + sizeof(int) * static_cast<size_t>(B) * nkv * kAttnCluster);
    L.ml = off;
    off = up256(off + sizeof(float2) * static_cast<size_t>(max_work) * nkv * rows_per_item);
    L.o = off;
    off = up256(off + sizeof(float) * static_cast<size_t>(max_work) * nkv * rows_per_item * D);
    L.total = off;
    return L;
}

// One block: clears the status word, builds the work list (one item per 1024-position group of
// every accepted sequence with a span), zeroes the group counters, and writes NaN rows for every
// sequence it rejects: a span longer than max_span (SDV_ERR_ARG) or one that passes max_context
// (SDV_ERR_CAPACITY) gets no work, so its rows would otherwise keep stale memory.
__global__ void noalloc_prep_kernel(const int *row_off, const int *base, int B, int nkv, int max_span,
                                    int max_context, int max_work, int *status, int *n_work, int4 *work,
                                    int *counters, bf16 *out, int row_elems) {
    pdl_wait();
    __shared__ int off_s[65];
    for (int i = threadIdx.x; i < B * nkv * kAttnCluster; i += blockDim.x) counters[i] = 0;
    if (threadIdx.x == 0) {
        *status = 0;
        int nw = 0;
        for (int b = 0; b < B; ++b) {
            const int S = row_off[b + 1] - row_off[b], L = base[b];
            off_s[b] = nw;
            if (S == 0) continue;
            if (S < 0 || S > max_span) {
                set_status(status, SDV_ERR_ARG);
                continue;
            }
            if (L < 0 || L + S > max_context) {
                set_status(status, SDV_ERR_CAPACITY);
                continue;
            }
            const int ng = (L + S + kAttnGroup - 1) / kAttnGroup;
            if (nw + ng > max_work) {
                set_status(status, SDV_ERR_CAPACITY);
                continue;
            }
            nw += ng;
        }
        off_s[B] = nw;
        *n_work = nw;
    }
    __syncthreads();
    for (int b = 0; b < B; ++b) {
        const int n = off_s[b + 1] - off_s[b];
        const int S = row_off[b + 1] - row_off[b];
        for (int g = threadIdx.x; g < n; g += blockDim.x) work[off_s[b] + g] = make_int4(b | (g << 16), base[b], S, row_off[b]);
        if (S > 0 && n == 0) {  // rejected sequence: its rows read as NaN rather than stale memory
            const size_t e0 = static_cast<size_t>(row_off[b]) * row_elems, e1 = static_cast<size_t>(row_off[b + 1]) * row_elems;
            for (size_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) out[e] = __float2bfloat16(NAN);
        }
    }
}

template <int D>
cudaError_t launch_attn(const AttnArgs &a, int max_work, int nkv, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(max_work * kAttnCluster, nkv);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = AttnShape<D>::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kAttnCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_kernel<D>, a);
}

// First call on a device: resolve the scratch array's device address (the host
// symbol is only a stand-in) and set the kernel attributes.
int setup_device(int dev, unsigned char **scratch) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SDV_ERR_CUDA;
        const cudaFuncAttribute smem = cudaFuncAttributeMaxDynamicSharedMemorySize;
        const cudaFuncAttribute carve = cudaFuncAttributePreferredSharedMemoryCarveout;
        if (cudaFuncSetAttribute(attn_kernel<128>, smem, AttnShape<128>::SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(attn_kernel<64>, smem, AttnShape<64>::SMEM) != cudaSuccess ||
            cudaFuncSetAttribute(attn_kernel<128>, carve, cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
            cudaFuncSetAttribute(attn_kernel<64>, carve, cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return SDV_ERR_CUDA;
        s.scratch = static_cast<unsigned char *>(p);
        s.done = true;
    }
    *scratch = s.scratch;
    return SDV_OK;
}

}  // namespace

extern "C" int sdv_paged_attention_noalloc(const void *d_q, const void *d_kv_layer, const int32_t *d_page_table,
                                           int pages_per_seq, int page_size, int n_pages, const int32_t *d_row_off,
                                           const int32_t *d_base, int B, int n_q_heads, int n_kv_heads,
                                           int head_dim, int max_span, int max_context, void *d_out,
                                           void *stream) {
    if (!d_q || !d_kv_layer || !d_page_table || !d_row_off || !d_base || !d_out) return SDV_ERR_ARG;
    if (B <= 0 || B > 64 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || page_size <= 0 ||
        n_pages <= 0 || pages_per_seq <= 0 || max_span <= 0 || max_context <= 0 ||
        max_context > pages_per_seq * page_size)
        return SDV_ERR_ARG;
    if (head_dim != 64 && head_dim != 128) return SDV_ERR_UNSUPPORTED;
    const int grp = n_q_heads / n_kv_heads;
    if (grp > 8 || 128 % grp) return SDV_ERR_UNSUPPORTED;
    // rows of one work item: grp heads x the span rows handled per launch
    const int qrows = std::min(max_span, kAttnRows / grp);
    const int max_work = B * ((max_context + kAttnGroup - 1) / kAttnGroup);
    const Layout L = layout(B, n_kv_heads, head_dim, grp * qrows, max_work);
    if (L.total > kScratchBytes) return SDV_ERR_CAPACITY;  // past the 8 MiB scratch: use sdv_op_attention

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDV_ERR_CUDA;
    unsigned char *scratch = nullptr;
    int r = setup_device(dev, &scratch);
    if (r) return r;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *status = reinterpret_cast<int *>(scratch);
    int *n_work = status + 1;
    int4 *work = reinterpret_cast<int4 *>(scratch + L.work);
    int *counters = reinterpret_cast<int *>(scratch + L.counters);
    noalloc_prep_kernel<<<1, 256, 0, st>>>(d_row_off, d_base, B, n_kv_heads, max_span, max_context, max_work, status,
                                            n_work, work, counters, static_cast<bf16 *>(d_out), n_q_heads * head_dim);
    if (cudaGetLastError() != cudaSuccess) return SDV_ERR_CUDA;

    AttnArgs a{};
    a.q = static_cast<const bf16 *>(d_q);
    a.q_plane = 0;
    a.out_plane = 0;
    a.kv_layer = static_cast<const bf16 *>(d_kv_layer);
    a.page_table = d_page_table;
    a.pages_per_seq = pages_per_seq;
    a.page_size = page_size;
    a.n_pages = n_pages;
    a.work = work;
    a.n_work = n_work;
    a.nq = n_q_heads;
    a.nkv = n_kv_heads;
    a.D = head_dim;
    a.grp = grp;
    a.qrows = qrows;
    a.scale_log2 = 1.4426950408889634f / std::sqrt(static_cast<float>(head_dim));
    a.part_o = reinterpret_cast<float *>(scratch + L.o);
    a.part_ml = reinterpret_cast<float2 *>(scratch + L.ml);
    a.counters = counters;
    a.out = static_cast<bf16 *>(d_out);
    a.status = status;
    for (int q0 = 0; q0 < max_span; q0 += qrows) {
        a.q0 = q0;
        const cudaError_t e = head_dim == 128 ? launch_attn<128>(a, max_work, n_kv_heads, st)
                                              : launch_attn<64>(a, max_work, n_kv_heads, st);
        if (e != cudaSuccess) return SDV_ERR_CUDA;
    }
    return SDV_OK;
}

extern "C" int sdv_noalloc_status(int32_t *h_status) {
    if (!h_status) return SDV_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDV_ERR_CUDA;
    unsigned char *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (g_setup[dev].done) scratch = g_setup[dev].scratch;
    }
    if (!scratch) {  // no call has run on this device: nothing to report
        *h_status = SDV_OK;
        return SDV_OK;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return SDV_ERR_CUDA;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpy(&v, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDV_ERR_CUDA;
    if (cudaMemcpy(scratch, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SDV_ERR_CUDA;
    *h_status = v;
    return SDV_OK;
}
