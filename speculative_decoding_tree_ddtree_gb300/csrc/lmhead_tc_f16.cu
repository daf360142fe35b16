// Instantiations of the fused lm_head + argmax kernel for f16 operands.
#include "lmhead_tc.cuh"

namespace lucetree {

namespace {

template <int RP>
cudaError_t launch_rp(const CUtensorMap& tw, const CUtensorMap& th, const lmhead::Args& a, int ctas,
                      cudaStream_t stream) {
    using Lay = lmhead::Layout<RP>;
    auto kern = lmhead::lmhead_kernel<false, RP>;
    static SmemLimitSeen seen;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), Lay::kBytes, seen);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(ctas), dim3(lmhead::kThreads), Lay::kBytes, stream, tw, th, a);
}

}  // namespace

cudaError_t launch_lmhead_f16(int rp, const CUtensorMap& tw, const CUtensorMap& th, const lmhead::Args& a, int ctas,
                               cudaStream_t stream) {
    switch (rp) {
        case 16: return launch_rp<16>(tw, th, a, ctas, stream);
        case 32: return launch_rp<32>(tw, th, a, ctas, stream);
        case 48: return launch_rp<48>(tw, th, a, ctas, stream);
        case 64: return launch_rp<64>(tw, th, a, ctas, stream);
        case 96: return launch_rp<96>(tw, th, a, ctas, stream);
        case 128: return launch_rp<128>(tw, th, a, ctas, stream);
        case 192: return launch_rp<192>(tw, th, a, ctas, stream);
        case 256: return launch_rp<256>(tw, th, a, ctas, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lucetree
