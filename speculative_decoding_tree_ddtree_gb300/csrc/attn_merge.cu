// attn_merge.cu -- the merge launch of lucetree_verify_attn: one CTA per
// output row (the routine is in attn_merge.cuh).
#include "attn_merge.cuh"

namespace lucetree {

namespace {

// Four warps per CTA = per output row, five CTAs per SM (at most 102
// registers a thread): a 528-row call then fits on the first 106 SMs that the
// prefix kernel frees, so its last blocks start early enough for their tree
// block to finish before the prefix kernel does.
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 5) merge_kernel(AttnLaunch L) {
    __shared__ float s_o[kWarps][D];
    __shared__ float s_red[kWarps];
    if (threadIdx.x == 0) pdl_trigger();
    const long long row = blockIdx.x;
    const int i = (int)((row / L.plan.Hq) % L.plan.N);
    const int b = (int)(row / ((long long)L.plan.Hq * L.plan.N));
    merge::merge_row<T, D, kWarps>(L, row, L.a.anc_mask[(size_t)b * L.plan.N + i], s_o, s_red);
}

}  // namespace

cudaError_t launch_attn_merge(const AttnLaunch& L, cudaStream_t stream) {
    const dim3 grid((unsigned)((long long)L.plan.B * L.plan.N * L.plan.Hq)), block(kThreads);
    if (L.a.dtype == LUCETREE_BF16) {
        if (L.a.D == 256) return launch_pdl(merge_kernel<__nv_bfloat16, 256>, grid, block, 0, stream, L);
        return launch_pdl(merge_kernel<__nv_bfloat16, 128>, grid, block, 0, stream, L);
    }
    if (L.a.D == 256) return launch_pdl(merge_kernel<__half, 256>, grid, block, 0, stream, L);
    return launch_pdl(merge_kernel<__half, 128>, grid, block, 0, stream, L);
}

}  // namespace lucetree
