// attn_prefix_simt.cu -- committed-prefix part of tree-verify attention on the
// CUDA cores: one warp per query row, streaming softmax over the CTA's key
// range, partial (O, max, sum) per split.  It follows the same split plan as
// the tensor-core kernel and exists as the simple reference path of the
// library's own kernels.
#include "internal.cuh"

namespace lucetree {

namespace {

__device__ inline float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ inline float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) prefix_simt_kernel(AttnLaunch L) {
    constexpr int DPL = D / 32;  // output dims per lane
    __shared__ float q_s[kWarps][D];
    const lucetree_attn_args& a = L.a;
    const PlanDims& p = L.plan;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, C = gridDim.x;

    const long long nT = total_tiles(p, a.ctx_len);
    if (nT == 0) return;
    const long long t0 = cta_begin(c, nT, C), t1 = cta_begin(c + 1, nT, C);
    if (t0 >= t1) return;

    const int per_seq = p.Hkv * p.rg.NG;
    const T* kpool = reinterpret_cast<const T*>(a.k_pool);
    const T* vpool = reinterpret_cast<const T*>(a.v_pool);
    const T* qg = reinterpret_cast<const T*>(a.q);
    long long off = 0;
    for (int s = 0; s < p.S && off < t1; ++s) {
        const int b = s / per_seq, g = (s % per_seq) / p.rg.NG, rg = s % p.rg.NG;
        const int Lb = seq_len(a.ctx_len, b, p.max_pages, (c == 0 && g == 0 && rg == 0) ? a.status : nullptr);
        const long long nt = tiles_of(Lb);
        const long long s0 = off, s1 = off + nt;
        off = s1;
        if (s1 <= t0 || nt == 0) continue;
        const int k0 = (int)((t0 > s0 ? t0 : s0) - s0) * kTileKeys;
        const int k1 = min((int)((t1 < s1 ? t1 : s1) - s0) * kTileKeys, Lb);
        float* slot = L.ws + (size_t)(c + s) * slot_floats(p);
        float* slot_m = slot + (size_t)p.rg.RG * D;
        float* slot_l = slot_m + p.rg.RG;
        const int i0 = rg * p.rg.NPG, i1 = min(p.N, i0 + p.rg.NPG);
        const int rows = (i1 - i0) * p.G;
        const int32_t* pt = a.page_table + (size_t)b * p.max_pages;

        for (int rl = warp; rl < rows; rl += kWarps) {
            const int i = i0 + rl / p.G, h = g * p.G + rl % p.G;
            const T* qrow = qg + (((size_t)b * p.N + i) * p.Hq + h) * D;
            for (int d = lane; d < D; d += 32) q_s[warp][d] = to_f32<T>(qrow[d]);
            __syncwarp();
            float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
            for (int x = 0; x < DPL; ++x) o[x] = 0.f;
            for (int kc = k0; kc < k1; kc += 32) {
                const int page = pt[kc / kPage];
                if (page < 0 || page >= a.num_pages) {
                    if (lane == 0) atomicOr(a.status, LUCETREE_DEV_BAD_PAGE);
                    continue;
                }
                const size_t page_base = ((size_t)page * p.Hkv + g) * kPage;
                const int key = kc + lane;
                const bool valid = key < k1;
                float sc = -INFINITY;
                if (valid) {
                    const T* krow = kpool + (page_base + (key % kPage)) * D;
                    float dot = 0.f;
#pragma unroll 4
                    for (int d = 0; d < D; d += 8) {
                        float kf[8];
                        load8_f32<T>(krow + d, kf);
#pragma unroll
                        for (int e = 0; e < 8; ++e) dot = fmaf(q_s[warp][d + e], kf[e], dot);
                    }
                    sc = dot * L.scale_log2;
                }
                const float mn = fmaxf(m, warp_max(sc));
                const float alpha = exp2f(m - mn);
                const float pj = valid ? exp2f(sc - mn) : 0.f;
                l = l * alpha + warp_sum(pj);
#pragma unroll
                for (int x = 0; x < DPL; ++x) o[x] *= alpha;
                const int cnt = min(32, k1 - kc);
                for (int j = 0; j < cnt; ++j) {
                    const float pjj = __shfl_sync(0xffffffffu, pj, j);
                    const T* vrow = vpool + (page_base + ((kc + j) % kPage)) * D + lane * DPL;
                    float vf[DPL];
                    if constexpr (DPL == 8) load8_f32<T>(vrow, vf);
                    else load4_f32<T>(vrow, vf);
#pragma unroll
                    for (int x = 0; x < DPL; ++x) o[x] = fmaf(pjj, vf[x], o[x]);
                }
                m = mn;
            }
#pragma unroll
            for (int x = 0; x < DPL; ++x) slot[(size_t)rl * D + lane * DPL + x] = o[x];
            if (lane == 0) {
                slot_m[rl] = m;
                slot_l[rl] = l;
            }
            __syncwarp();
        }
    }
}

}  // namespace

int prefix_grid_ctas(int device) { return device_sm_count(device) * 2; }

cudaError_t launch_attn_prefix(const AttnLaunch& L, cudaStream_t stream) {
    dim3 grid(L.plan.C), block(kWarps * 32);
    if (L.a.dtype == LUCETREE_BF16) {
        if (L.a.D == 256) prefix_simt_kernel<__nv_bfloat16, 256><<<grid, block, 0, stream>>>(L);
        else prefix_simt_kernel<__nv_bfloat16, 128><<<grid, block, 0, stream>>>(L);
    } else {
        if (L.a.D == 256) prefix_simt_kernel<__half, 256><<<grid, block, 0, stream>>>(L);
        else prefix_simt_kernel<__half, 128><<<grid, block, 0, stream>>>(L);
    }
    return cudaGetLastError();
}

}  // namespace lucetree
