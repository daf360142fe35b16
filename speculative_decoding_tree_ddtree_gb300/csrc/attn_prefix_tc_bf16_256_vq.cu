// Instantiations of the tensor-core prefix kernel for bf16 operands, head dim 256, with V held as
// int8 or int4 codes and per-token power-of-two exponents; dispatch over the V format.
#include "attn_prefix_tc.cuh"

namespace lucetree {

cudaError_t launch_prefix_tc_bf16_256_v16(int rgp, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                                          const AttnLaunch& L, cudaStream_t stream);

cudaError_t launch_prefix_tc_bf16_256(int rgp, int vq, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const CUtensorMap& tq, const CUtensorMap& tve, const AttnLaunch& L,
                                      cudaStream_t stream) {
    if (vq == 1) return prefix_tc::launch_rgp<256, true, 1>(rgp, tk, tv, tq, tve, tv, L, stream);
    if (vq == 2) return prefix_tc::launch_rgp<256, true, 2>(rgp, tk, tv, tq, tve, tv, L, stream);
    return launch_prefix_tc_bf16_256_v16(rgp, tk, tv, tq, L, stream);
}

}  // namespace lucetree
