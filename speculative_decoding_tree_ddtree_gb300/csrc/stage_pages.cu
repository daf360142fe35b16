// stage_pages.cu -- host-resident cold KV pages staged into the device pool.
//
// The pages keep cold 64-token chunks in host memory and bring them back to
// the GPU for attention ("Lucebox Hub", section "KVFlash").  Here the caller
// keeps host-resident K and V pools ([host_pages][Hkv][64][D], page-locked) and
// asks for a list of them to be copied into free device pool pages before
// the verify step; the kernel reads host memory directly over the CPU-GPU
// link (zero copy: 16-byte loads from the mapped host pages, several in
// flight per thread) and writes the device pool, then points the listed
// page-table entries at the new pages.  Attention itself is unchanged: it
// only ever reads the device pool.
#include "internal.cuh"
#include "stage.h"

namespace lucetree {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct StageLaunch {
    lucetree_stage_args a;
    const uint4* hk;  // device-visible addresses of the host pools
    const uint4* hv;
    long long units_per_page;  // 16-byte units of one page of one tensor
};

__global__ void __launch_bounds__(kThreads) stage_kernel(StageLaunch L) {
    const lucetree_stage_args& a = L.a;
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) pdl_trigger();
    const long long upp = L.units_per_page;
    const long long total = 2ll * a.n * upp;  // K pages then V pages
    const long long stride = (long long)gridDim.x * kThreads;
    uint4* kp = reinterpret_cast<uint4*>(a.k_pool);
    uint4* vp = reinterpret_cast<uint4*>(a.v_pool);
    for (long long e0 = (long long)blockIdx.x * kThreads + threadIdx.x; e0 < total; e0 += kUnroll * stride) {
        uint4 x[kUnroll];
        uint4* to[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long e = e0 + u * stride;
            to[u] = nullptr;
            if (e < total) {
                const bool is_v = e >= (long long)a.n * upp;
                const long long f = is_v ? e - (long long)a.n * upp : e;
                const int i = (int)(f / upp);
                const long long w = f % upp;
                const int s = a.src[i], d = a.dst[i];
                if (s < 0 || s >= a.host_pages || d < 0 || d >= a.num_pages) {
                    if (w == 0 && !is_v) atomicOr(a.status, LUCETREE_DEV_BAD_PAGE);
                    continue;
                }
                x[u] = (is_v ? L.hv : L.hk)[(long long)s * upp + w];
                to[u] = (is_v ? vp : kp) + (long long)d * upp + w;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (to[u]) *to[u] = x[u];
    }
    if (a.table_idx) {
        for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < a.n; i += stride) {
            const int t = a.table_idx[i], d = a.dst[i];
            if (t < 0 || t >= a.table_len || d < 0 || d >= a.num_pages) {
                atomicOr(a.status, LUCETREE_DEV_BAD_PAGE);
                continue;
            }
            a.page_table[t] = d;
        }
    }
}

}  // namespace

cudaError_t launch_stage_pages(const lucetree_stage_args& a, const void* host_k_dev, const void* host_v_dev,
                               cudaStream_t stream) {
    if (a.n == 0) return cudaSuccess;
    StageLaunch L;
    L.a = a;
    L.hk = reinterpret_cast<const uint4*>(host_k_dev);
    L.hv = reinterpret_cast<const uint4*>(host_v_dev);
    L.units_per_page = (long long)a.Hkv * kPage * a.D * 2 / 16;
    int dev = 0;
    cudaGetDevice(&dev);
    const long long total = 2ll * a.n * L.units_per_page;
    long long ctas = (total + (long long)kThreads * kUnroll - 1) / ((long long)kThreads * kUnroll);
    const long long cap = 4ll * device_sm_count(dev);
    if (ctas > cap) ctas = cap;
    if (ctas < 1) ctas = 1;
    return launch_pdl(stage_kernel, dim3((unsigned)ctas), dim3(kThreads), 0, stream, L);
}

}  // namespace lucetree
