// attn_merge.cu -- tree block + log-sum-exp merge of tree-verify attention.
//
// One warp per output row (b, node i, head h).  The warp runs the softmax
// over the tree keys j with bit j of anc_mask[b][i] set (the node's ancestors
// and itself), then folds in the prefix partials (O, max, sum) that the
// split-K prefix kernel left for this row's segment, and writes
// out = O / sum and lse = ln(sum) + max.  Maxima are kept in the log2 domain
// (scores pre-multiplied by log2 e), so every rescale is one exp2.
//
// The split partials are independent, so the warp reads their maxima and sums
// with one lane per split, forms every split's weight once, and then adds the
// weighted partial rows with several loads in flight instead of walking the
// splits one dependent load at a time.
#include "internal.cuh"

namespace lucetree {

namespace {

__device__ inline float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ inline float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

constexpr int kRowsPerBlock = 4;
constexpr int kBatch = 8;  // partial rows in flight per lane

template <typename T, int D>
__device__ inline void load_slice(const T* p, float (&out)[D / 32]) {
    if constexpr (D / 32 == 8) load8_f32<T>(p, out);
    else load4_f32<T>(p, out);
}

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

    float qf[DPL];
    load_slice<T, D>(reinterpret_cast<const T*>(a.q) + (size_t)row * D + lane * DPL, qf);

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
        load_slice<T, D>(kt + base, kf);
        load_slice<T, D>(vt + base, vf);
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
        const int count = c_hi - c_lo + 1;
        const size_t sf = slot_floats(p);
        const size_t slot0 = slot_index(p, rg, c_lo, s);
        const float* ws = L.ws;
        // with fewer tiles than CTAs some CTAs own no tile and write no partial
        auto weight_of = [&](int k, float& mk, float& lk) {
            const int c = c_lo + k;
            mk = -INFINITY;
            lk = 0.f;
            if (k < count && cta_begin(c, nT, p.Cg) != cta_begin(c + 1, nT, p.Cg)) {
                const float* slot = ws + (slot0 + k) * sf + (size_t)p.rg.RG * D;
                mk = slot[rl];
                lk = slot[p.rg.RG + rl];
            }
        };
        // pass 1: the common shift and the sum, one lane per split
        float mmax = m;
        for (int k0 = 0; k0 < count; k0 += 32) {
            float mk, lk;
            weight_of(k0 + lane, mk, lk);
            mmax = fmaxf(mmax, warp_max(mk));
        }
        const float a_tree = m > -INFINITY ? exp2f(m - mmax) : 0.f;
        float lsum = 0.f;
#pragma unroll
        for (int x = 0; x < DPL; ++x) o[x] *= a_tree;
        // pass 2: weighted partial rows, kBatch loads in flight
        for (int k0 = 0; k0 < count; k0 += 32) {
            float mk, lk;
            weight_of(k0 + lane, mk, lk);
            const float wk = mk > -INFINITY ? exp2f(mk - mmax) : 0.f;
            lsum += wk * lk;
            const int n = min(32, count - k0);
            for (int e0 = 0; e0 < n; e0 += kBatch) {
                float w[kBatch];
                float part[kBatch][DPL];
#pragma unroll
                for (int e = 0; e < kBatch; ++e) {
                    w[e] = __shfl_sync(0xffffffffu, wk, (e0 + e) & 31);
                    if (e0 + e < n && w[e] != 0.f) {
                        const float* op = ws + (slot0 + k0 + e0 + e) * sf + (size_t)rl * D + lane * DPL;
                        if constexpr (DPL == 8) {
                            const float4 v0 = *reinterpret_cast<const float4*>(op);
                            const float4 v1 = *reinterpret_cast<const float4*>(op + 4);
                            part[e][0] = v0.x; part[e][1] = v0.y; part[e][2] = v0.z; part[e][3] = v0.w;
                            part[e][4] = v1.x; part[e][5] = v1.y; part[e][6] = v1.z; part[e][7] = v1.w;
                        } else {
                            const float4 v0 = *reinterpret_cast<const float4*>(op);
                            part[e][0] = v0.x; part[e][1] = v0.y; part[e][2] = v0.z; part[e][3] = v0.w;
                        }
                    } else {
                        w[e] = 0.f;
#pragma unroll
                        for (int x = 0; x < DPL; ++x) part[e][x] = 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < kBatch; ++e)
#pragma unroll
                    for (int x = 0; x < DPL; ++x) o[x] = fmaf(part[e][x], w[e], o[x]);
            }
        }
        l = l * a_tree + warp_sum(lsum);
        m = mmax;
    }

    const float inv = 1.f / l;
    float* orow = a.out + (size_t)row * D + lane * DPL;
#pragma unroll
    for (int x = 0; x < DPL; x += 4)
        *reinterpret_cast<float4*>(orow + x) = make_float4(o[x] * inv, o[x + 1] * inv, o[x + 2] * inv, o[x + 3] * inv);
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
