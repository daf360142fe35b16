// Instantiations of the tensor-core prefix kernel with K held as FP8 E4M3 codes (bf16 queries,
// head dim 256) and V as int4 codes with per-token exponents.
#include "attn_prefix_tc.cuh"

namespace lucetree {

cudaError_t launch_prefix_tc_bf16_256_kq_v4(int rgp, const CUtensorMap& tk, const CUtensorMap& tv,
                                            const CUtensorMap& tq, const CUtensorMap& tve, const CUtensorMap& tq2,
                                            const AttnLaunch& L, cudaStream_t stream) {
    return prefix_tc::launch_rgp<256, true, 2, 1>(rgp, tk, tv, tq, tve, tq2, L, stream);
}

cudaError_t launch_prefix_tc_bf16_256_kq_v16(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const CUtensorMap&, const CUtensorMap&, const AttnLaunch&, cudaStream_t);
cudaError_t launch_prefix_tc_bf16_256_kq_v8(int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const CUtensorMap&, const AttnLaunch&, cudaStream_t);

// dispatch over the V format (0 = bf16, 1 = int8 codes, 2 = int4 codes)
cudaError_t launch_prefix_tc_bf16_256_kq(int rgp, int vq, const CUtensorMap& tk, const CUtensorMap& tv,
                                         const CUtensorMap& tq, const CUtensorMap& tve, const CUtensorMap& tq2,
                                         const AttnLaunch& L, cudaStream_t stream) {
    if (vq == 1) return launch_prefix_tc_bf16_256_kq_v8(rgp, tk, tv, tq, tve, tq2, L, stream);
    if (vq == 2) return launch_prefix_tc_bf16_256_kq_v4(rgp, tk, tv, tq, tve, tq2, L, stream);
    return launch_prefix_tc_bf16_256_kq_v16(rgp, tk, tv, tq, tve, tq2, L, stream);
}

}  // namespace lucetree
