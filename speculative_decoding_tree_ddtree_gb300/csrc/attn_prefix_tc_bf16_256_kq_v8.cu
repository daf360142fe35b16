// Instantiations of the tensor-core prefix kernel with K held as FP8 E4M3 codes (bf16 queries,
// head dim 256) and V as int8 codes with per-token exponents.
#include "attn_prefix_tc.cuh"

namespace lucetree {

cudaError_t launch_prefix_tc_bf16_256_kq_v8(int rgp, const CUtensorMap& tk, const CUtensorMap& tv,
                                            const CUtensorMap& tq, const CUtensorMap& tve, const CUtensorMap& tq2,
                                            const AttnLaunch& L, cudaStream_t stream) {
    return prefix_tc::launch_rgp<256, true, 1, 1>(rgp, tk, tv, tq, tve, tq2, L, stream);
}

}  // namespace lucetree
