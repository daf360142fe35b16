// tree_ops.cu -- ancestor masks, greedy acceptance and the commit copy (the
// acceptance and commit routines are in tree_ops.cuh).
#include "tree_ops.cuh"

namespace lucetree {

namespace {

// One warp per sequence; node i lives in lane i % 32, slot i / 32.  Parents
// are loaded in parallel, then the masks are built in node order (each node
// needs its parent's mask) with shuffles instead of dependent global loads.
__global__ void __launch_bounds__(128) build_anc_kernel(const int32_t* __restrict__ parent, int B, int N,
                                                        uint64_t* __restrict__ anc, uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int32_t* par = parent + (size_t)b * N;
    int p0 = lane < N ? par[lane] : -1;
    int p1 = lane + 32 < N ? par[lane + 32] : -1;
    uint64_t m0 = 0, m1 = 0;  // this lane's nodes' masks
    bool bad = false;
    for (int i = 0; i < N; ++i) {
        const int pi = __shfl_sync(0xffffffffu, i < 32 ? p0 : p1, i & 31);
        uint64_t pm = 0;
        if (pi >= 0 && pi < i) {
            const uint64_t a0 = __shfl_sync(0xffffffffu, m0, pi & 31);
            const uint64_t a1 = __shfl_sync(0xffffffffu, m1, pi & 31);
            pm = pi < 32 ? a0 : a1;
        } else if (pi != -1) {
            bad = true;
        }
        const uint64_t mi = pm | (1ull << i);
        if ((i & 31) == lane) {
            if (i < 32) m0 = mi;
            else m1 = mi;
        }
    }
    uint64_t* out = anc + (size_t)b * N;
    if (lane < N) out[lane] = m0;
    if (lane + 32 < N) out[lane + 32] = m1;
    if (bad && lane == 0) atomicOr(status, LUCETREE_DEV_BAD_PARENT);
}

// One warp per sequence (the routine is in tree_ops.cuh).
__global__ void __launch_bounds__(128) accept_kernel(const int32_t* __restrict__ parent,
                                                     const int32_t* __restrict__ draft,
                                                     const int32_t* __restrict__ argmax, int B, int N, int vocab,
                                                     int32_t* __restrict__ acc_nodes, int32_t* __restrict__ acc_len,
                                                     int32_t* __restrict__ bonus, uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (b >= B) return;
    tree::accept_warp(parent + (size_t)b * N, draft + (size_t)b * N, argmax + (size_t)b * (N + 1), N, vocab,
                      acc_nodes + (size_t)b * N, acc_len + b, bonus + b, status);
}

// One CTA per sequence (the routine is in tree_ops.cuh).
__global__ void __launch_bounds__(256) commit_kernel(lucetree_commit_args c, int elem_bytes) {
    __shared__ int s_good;
    pdl_wait();
    pdl_trigger();
    tree::commit_block(c, blockIdx.x, elem_bytes, &s_good);
}

}  // namespace

cudaError_t launch_build_anc(const int32_t* parent, int B, int N, uint64_t* anc, uint32_t* status,
                             cudaStream_t stream) {
    return launch_pdl(build_anc_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, parent, B, N, anc, status);
}

cudaError_t launch_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int B, int N,
                          int vocab, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, uint32_t* status,
                          cudaStream_t stream) {
    return launch_pdl(accept_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, parent, draft, argmax, B, N, vocab,
                      acc_nodes, acc_len, bonus, status);
}

cudaError_t launch_commit(const lucetree_commit_args& c, cudaStream_t stream) {
    return launch_pdl(commit_kernel, dim3(c.B), dim3(256), 0, stream, c, 2);
}

}  // namespace lucetree
