// Instantiations of the tensor-core prefix kernel for f16 operands, head dim 128.
#include "attn_prefix_tc.cuh"

namespace lucetree {

cudaError_t launch_prefix_tc_f16_128(int rgp, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                                     const AttnLaunch& L, cudaStream_t stream) {
    return prefix_tc::launch_rgp<128, false>(rgp, tk, tv, tq, tv, tv, L, stream);
}

}  // namespace lucetree
