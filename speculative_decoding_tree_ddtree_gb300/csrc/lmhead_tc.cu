// lmhead_tc.cu -- host side of the fused lm_head + argmax: TMA tensor maps over
// the weight and the hidden states, padded row count, grid size.
#include <cuda.h>

#include "lmhead_tc.cuh"
#include "lmhead.h"

namespace lucetree {

// padded row count: the smallest instantiated multiple of 16 >= rows
int lmhead_padded_rows(int rows) {
    static const int kRP[] = {16, 32, 48, 64, 96, 128, 192, 256};
    for (int rp : kRP)
        if (rows <= rp) return rp;
    return -1;
}

size_t lmhead_workspace_bytes(int rows) { return ((size_t)rows * 8 + 255) / 256 * 256 + 256; }

cudaError_t launch_lmhead(const lucetree_lmhead_args& a, void* ws, cudaStream_t stream) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const CUtensorMapDataType dt =
        a.dtype == LUCETREE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int rp = lmhead_padded_rows(a.rows);
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap tw, th;
    // weight [vocab][d_model]; box = 64 dims x 128 vocabulary rows (128-byte swizzle)
    const cuuint64_t w_dims[2] = {(cuuint64_t)a.d_model, (cuuint64_t)a.vocab};
    const cuuint64_t w_strides[1] = {(cuuint64_t)a.d_model * 2};
    const cuuint32_t w_box[2] = {64, (cuuint32_t)lmhead::kVT};
    if (enc(&tw, dt, 2, const_cast<void*>(a.weight), w_dims, w_strides, w_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // hidden [rows][d_model]; box = 64 dims x rp rows (rows past `rows` read as zero)
    const cuuint64_t h_dims[2] = {(cuuint64_t)a.d_model, (cuuint64_t)a.rows};
    const cuuint64_t h_strides[1] = {(cuuint64_t)a.d_model * 2};
    const cuuint32_t h_box[2] = {64, (cuuint32_t)rp};
    if (enc(&th, dt, 2, const_cast<void*>(a.hidden), h_dims, h_strides, h_box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    lmhead::Args k;
    k.rows = a.rows;
    k.d_model = a.d_model;
    k.vocab = a.vocab;
    k.keys = reinterpret_cast<unsigned long long*>(ws);
    k.ticket = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(ws) + ((size_t)a.rows * 8 + 255) / 256 * 256);
    k.out_idx = a.out_idx;
    k.out_logit = a.out_logit;
    k.status = a.status;
    // keys and ticket start at zero (the kernel also leaves them zero)
    cudaError_t e = cudaMemsetAsync(ws, 0, lmhead_workspace_bytes(a.rows), stream);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    const int n_tiles = (a.vocab + lmhead::kVT - 1) / lmhead::kVT;
    const int slots = device_sm_count(dev) * lmhead::ctas_per_sm(rp);
    const int ctas = n_tiles < slots ? n_tiles : slots;
    return a.dtype == LUCETREE_BF16 ? launch_lmhead_bf16(rp, tw, th, k, ctas, stream)
                                    : launch_lmhead_f16(rp, tw, th, k, ctas, stream);
}

}  // namespace lucetree
