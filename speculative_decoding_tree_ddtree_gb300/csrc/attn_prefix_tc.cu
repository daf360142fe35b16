// attn_prefix_tc.cu -- host side of the tensor-core prefix kernel: TMA tensor
// maps over the K/V pools and the queries, kernel selection by head dim,
// operand type and padded row count.
#include <cuda.h>

#include "attn_prefix_tc.cuh"

namespace lucetree {

int prefix_grid_ctas(int device) { return device_sm_count(device); }

bool prefix_shape_supported(const lucetree_attn_args& a) {
    // TMA row coordinates are 32-bit: the pool must stay below 2^31 rows
    const long long rows = (long long)a.num_pages * a.Hkv * kPage;
    // the kernel counts key tiles in 32 bits
    const long long tiles = (long long)a.B * a.Hkv * (((long long)a.max_pages_per_seq * kPage + kTileKeys - 1) / kTileKeys);
    return rows + kPage < (1ll << 31) && tiles < (1ll << 31);
}

cudaError_t launch_attn_prefix(const AttnLaunch& L, cudaStream_t stream) {
    const lucetree_attn_args& a = L.a;
    const PlanDims& p = L.plan;
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        a.dtype == LUCETREE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint32_t estr[3] = {1, 1, 1};

    // K, V pools as 2-D [num_pages * Hkv * 64 rows][D]; box = one 64-token page x 64 dims
    // (E4M3 K: codes as bytes [rows][D], box = one page x 128 dims)
    const bool kq = L.k_format == LUCETREE_K_E4M3;
    CUtensorMap tk, tv, tq, tq2;
    const cuuint64_t kv_dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.num_pages * a.Hkv * kPage};
    const cuuint64_t kv_strides[1] = {(cuuint64_t)a.D * 2};
    const cuuint32_t kv_box[2] = {64, (cuuint32_t)kPage};
    const cuuint64_t kc_strides[1] = {(cuuint64_t)a.D};
    const cuuint32_t kc_box[2] = {128, (cuuint32_t)kPage};
    if (enc(&tk, kq ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : dt, 2, const_cast<void*>(a.k_pool), kv_dims,
            kq ? kc_strides : kv_strides, kq ? kc_box : kv_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (enc(&tv, dt, 2, const_cast<void*>(a.v_pool), kv_dims, kv_strides, kv_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // queries as 3-D [B*N nodes][Hq heads][D]; box = 64 dims x G heads x NPG nodes
    const cuuint64_t q_dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.N};
    const cuuint64_t q_strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.Hq * a.D * 2};
    const cuuint32_t q_box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)p.rg.NPG};
    // (E4M3 K too: the kernel splits the bf16 queries into their two E4M3 parts on chip)
    if (enc(&tq, dt, 3, const_cast<void*>(a.q), q_dims, q_strides, q_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    tq2 = tv;

    // quantised V: codes as bytes [rows][D or D/2] (one 64-token page x 128 dims per box, no
    // swizzle: the softmax warps expand them), exponents [num_pages * Hkv][64] one page per box
    const int vq = L.v_format == LUCETREE_V_INT8 ? 1 : (L.v_format == LUCETREE_V_INT4 ? 2 : 0);
    CUtensorMap tve = tv;
    if (vq) {
        const cuuint64_t row_bytes = vq == 1 ? (cuuint64_t)a.D : (cuuint64_t)a.D / 2;
        const cuuint64_t c_dims[2] = {row_bytes, (cuuint64_t)a.num_pages * a.Hkv * kPage};
        const cuuint64_t c_strides[1] = {row_bytes};
        const cuuint32_t c_box[2] = {vq == 1 ? 128u : 64u, (cuuint32_t)kPage};
        if (enc(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(a.v_pool), c_dims, c_strides, c_box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        const cuuint64_t e_dims[2] = {(cuuint64_t)kPage, (cuuint64_t)a.num_pages * a.Hkv};
        const cuuint64_t e_strides[1] = {(cuuint64_t)kPage};
        const cuuint32_t e_box[2] = {(cuuint32_t)kPage, 1};
        if (enc(&tve, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(L.v_exp), e_dims, e_strides, e_box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const int rgp = (p.rg.RG + 15) / 16 * 16;
    if (kq) return launch_prefix_tc_bf16_256_kq(rgp, vq, tk, tv, tq, tve, tq2, L, stream);
    if (a.dtype == LUCETREE_BF16)
        return a.D == 256 ? launch_prefix_tc_bf16_256(rgp, vq, tk, tv, tq, tve, L, stream)
                          : launch_prefix_tc_bf16_128(rgp, tk, tv, tq, L, stream);
    return a.D == 256 ? launch_prefix_tc_f16_256(rgp, vq, tk, tv, tq, tve, L, stream)
                      : launch_prefix_tc_f16_128(rgp, tk, tv, tq, L, stream);
}

}  // namespace lucetree
