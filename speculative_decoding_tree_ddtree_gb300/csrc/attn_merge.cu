// attn_merge.cu -- tree block + log-sum-exp merge of tree-verify attention.
//
// One warp per output row (b, node i, head h).  The warp first runs the
// softmax over the tree keys j with bit j of anc_mask[b][i] set (the node's
// ancestors and itself), then folds in the prefix partials (O, max, sum) that
// the split-K prefix kernel left for this row's segment, and writes
// out = O / sum and lse = ln(sum) + max.  Maxima are kept in the log2 domain
// (scores pre-multiplied by log2 e), so every rescale is one exp2.
#include "internal.cuh"

namespace lucetree {

namespace {

__device__ inline float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kRowsPerBlock = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32) merge_kernel(AttnLaunch L) {
    constexpr int DPL = D / 32;
    const lucetree_attn_args& a = L.a;
    const PlanDims& p = L.plan;
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    const long long total_rows = (long long)p.B * p.N * p.Hq;
    if (row >= total_rows) return;
    const int h = (int)(row % p.Hq);
    const int i = (int)((row / p.Hq) % p.N);
    const int b = (int)(row / ((long long)p.Hq * p.N));
    const int g = h / p.G;
    const int rg = i / p.rg.NPG;
    const int rl = (i - rg * p.rg.NPG) * p.G + (h % p.G);
    const int s = b * p.Hkv + g;

    const T* qrow = reinterpret_cast<const T*>(a.q) + (size_t)row * D + lane * DPL;
    float qf[DPL];
    if constexpr (DPL == 8) load8_f32<T>(qrow, qf);
    else load4_f32<T>(qrow, qf);

    // ---- tree block: keys of the node's ancestors and itself
    uint64_t anc = a.anc_mask[(size_t)b * p.N + i];
    if (p.N < 64) anc &= (1ull << p.N) - 1ull;
    if (!((anc >> i) & 1ull) && lane == 0) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int x = 0; x < DPL; ++x) o[x] = 0.f;
    const T* kt = reinterpret_cast<const T*>(a.k_tree);
    const T* vt = reinterpret_cast<const T*>(a.v_tree);
    while (anc) {
        const int j = __ffsll((long long)anc) - 1;
        anc &= anc - 1ull;
        const size_t base = (((size_t)b * p.N + j) * p.Hkv + g) * D + lane * DPL;
        float kf[DPL], vf[DPL];
        if constexpr (DPL == 8) {
            load8_f32<T>(kt + base, kf);
            load8_f32<T>(vt + base, vf);
        } else {
            load4_f32<T>(kt + base, kf);
            load4_f32<T>(vt + base, vf);
        }
        float dot = 0.f;
#pragma unroll
        for (int x = 0; x < DPL; ++x) dot = fmaf(qf[x], kf[x], dot);
        const float sc = warp_sum(dot) * L.scale_log2;
        const float mn = fmaxf(m, sc);
        const float alpha = exp2f(m - mn), pj = exp2f(sc - mn);
        l = l * alpha + pj;
#pragma unroll
        for (int x = 0; x < DPL; ++x) o[x] = fmaf(o[x], alpha, pj * vf[x]);
        m = mn;
    }

    // ---- committed prefix: partials of every CTA that covered this segment
    const int Lb = seq_len(a.ctx_len, b, p.max_pages, (i == 0 && h == 0 && lane == 0) ? a.status : nullptr);
    if (Lb > 0) {
        const long long nT = total_tiles(p, a.ctx_len);
        const long long first = segment_offset(p, a.ctx_len, s);
        const long long last = first + tiles_of(Lb) - 1;
        const int c_lo = cta_of_tile(first, nT, p.Cg), c_hi = cta_of_tile(last, nT, p.Cg);
        for (int c = c_lo; c <= c_hi; ++c) {
            // with fewer tiles than CTAs some CTAs own no tile and write no partial
            if (cta_begin(c, nT, p.Cg) == cta_begin(c + 1, nT, p.Cg)) continue;
            const float* slot = L.ws + slot_index(p, rg, c, s) * slot_floats(p);
            const float mp = slot[(size_t)p.rg.RG * D + rl];
            const float lp = slot[(size_t)p.rg.RG * D + p.rg.RG + rl];
            if (!(mp > -INFINITY)) continue;  // split saw no valid key
            const float mn = fmaxf(m, mp);
            const float a1 = exp2f(m - mn), a2 = exp2f(mp - mn);
            l = l * a1 + lp * a2;
            const float* op = slot + (size_t)rl * D + lane * DPL;
#pragma unroll
            for (int x = 0; x < DPL; ++x) o[x] = fmaf(o[x], a1, op[x] * a2);
            m = mn;
        }
    }

    const float inv = 1.f / l;
    float* orow = a.out + (size_t)row * D + lane * DPL;
#pragma unroll
    for (int x = 0; x < DPL; ++x) orow[x] = o[x] * inv;
    if (a.lse && lane == 0) a.lse[row] = (m + log2f(l)) * kLn2;
}

}  // namespace

cudaError_t launch_attn_merge(const AttnLaunch& L, cudaStream_t stream) {
    const long long rows = (long long)L.plan.B * L.plan.N * L.plan.Hq;
    dim3 grid((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock)), block(kRowsPerBlock * 32);
    if (L.a.dtype == LUCETREE_BF16) {
        if (L.a.D == 256) merge_kernel<__nv_bfloat16, 256><<<grid, block, 0, stream>>>(L);
        else merge_kernel<__nv_bfloat16, 128><<<grid, block, 0, stream>>>(L);
    } else {
        if (L.a.D == 256) merge_kernel<__half, 256><<<grid, block, 0, stream>>>(L);
        else merge_kernel<__half, 128><<<grid, block, 0, stream>>>(L);
    }
    return cudaGetLastError();
}

}  // namespace lucetree
