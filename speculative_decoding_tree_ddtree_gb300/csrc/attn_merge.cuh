// attn_merge.cuh -- tree block + log-sum-exp merge of tree-verify attention,
// as a CTA device routine shared by the merge kernel and the fused step.
//
// One group of four warps per output row (b, node i, head h).  The warps share the softmax
// over the tree keys j with bit j of anc_mask[b][i] set (the node's ancestors
// and itself) and the prefix partials (O, max, sum) that the split-K prefix
// kernel left for this row's key segment; the block writes out = O / sum and
// lse = ln(sum) + max.  Maxima are kept in the log2 domain
// (scores pre-multiplied by log2 e), so every rescale is one exp2.
//
// The partials are independent: warp w folds partials w, w + 4, ... into a
// running (max, sum, output slice) of its own, issuing all of a round's
// loads before using any, and the four warps' parts are combined through
// shared memory on their common maximum.  A row reads about 40 partial rows
// of D floats, so spreading them over four warps, five rows a round, gets the
// whole row in about two L2 round trips instead of one dependent row at a
// time.
#pragma once

#include "internal.cuh"

namespace lucetree {

namespace merge {

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

// Four warps per output row, in the merge launch (one 128-thread CTA per row,
// up to five CTAs per SM, so a 528-row call fits in one wave) and in the fused
// step's finish kernel (two rows per 256-thread CTA), so both give the same
// bits.  Each warp folds its partials in rounds of kRound rows, all loads of a
// round in flight together.
constexpr int kRound = 5;
constexpr int kMaxTreeBatch = 2;  // ancestors whose K/V a warp loads before using any (registers)

template <typename T, int D>
__device__ inline void load_slice(const T* p, float (&out)[D / 32]) {
    if constexpr (D / 32 == 8) load8_f32<T>(p, out);
    else load4_f32<T>(p, out);
}

template <int DPL>
__device__ inline void load_partial(const float* op, float (&v)[DPL]) {
    const float4 a = *reinterpret_cast<const float4*>(op);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    if constexpr (DPL == 8) {
        const float4 b = *reinterpret_cast<const float4*>(op + 4);
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}


__device__ __forceinline__ void group_sync(int bar_id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(threads) : "memory");
}

// One output row (b, node i, head h) by a group of W warps starting at warp
// wbase of the CTA, which synchronise on named barrier bar_id (so several
// groups of a CTA can each merge a row).  anc: the node's ancestor-or-self
// mask.  s_o: W x D floats and s_red: W floats of shared memory (the
// group's own).  Runs the tree block, then pdl_wait(), then the log-sum-exp
// merge of the prefix partials.  The arithmetic depends only on W.
template <typename T, int D, int W, int kBar = 1>
__device__ __forceinline__ void merge_row(const AttnLaunch& L, long long row, uint64_t anc, float (*s_o)[D],
                                          float* s_red, int wbase = 0) {
    constexpr int bar_id = kBar;
    constexpr int DPL = D / 32;
    constexpr int kR = kRound;
    const lucetree_attn_args& a = L.a;
    const PlanDims& p = L.plan;
    const int gt = threadIdx.x - 32 * wbase;  // thread index within the group
    const int warp = gt >> 5, lane = threadIdx.x & 31;
    const int h = (int)(row % p.Hq);
    const int i = (int)((row / p.Hq) % p.N);
    const int b = (int)(row / ((long long)p.Hq * p.N));
    const int g = h / p.G;
    const int rg = i / p.rg.NPG;
    const int rl = (i - rg * p.rg.NPG) * p.G + (h % p.G);
    const int s = b * p.Hkv + g;

    // ---- tree block: keys of the node's ancestors and itself, the k-th such
    // key (in node order) handled by warp k % W with its own running max, sum
    // and output slice; a warp loads the K/V slices of up to kMaxTreeBatch of
    // its keys before using any
    float o[DPL];
#pragma unroll
    for (int x = 0; x < DPL; ++x) o[x] = 0.f;
    float m_t = -INFINITY, l_t = 0.f;
    {
        float qf[DPL];
        load_slice<T, D>(reinterpret_cast<const T*>(a.q) + (size_t)row * D + lane * DPL, qf);
        if (p.N < 64) anc &= (1ull << p.N) - 1ull;
        if (!((anc >> i) & 1ull) && gt == 0) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
        // this warp's keys: every W-th set bit of anc, starting at rank `warp`
        uint64_t mine = 0;
        {
            uint64_t rest = anc;
            int rank = 0;
            while (rest) {
                const int j = __ffsll((long long)rest) - 1;
                rest &= rest - 1ull;
                if ((rank++ % W) == warp) mine |= 1ull << j;
            }
        }
        const T* kt = reinterpret_cast<const T*>(a.k_tree);
        const T* vt = reinterpret_cast<const T*>(a.v_tree);
        while (mine) {
            int js[kMaxTreeBatch];
            int nb = 0;
#pragma unroll
            for (int u = 0; u < kMaxTreeBatch; ++u) {
                js[u] = -1;
                if (mine) {
                    js[u] = __ffsll((long long)mine) - 1;
                    mine &= mine - 1ull;
                    ++nb;
                }
            }
            float kf[kMaxTreeBatch][DPL], vf[kMaxTreeBatch][DPL];
#pragma unroll
            for (int u = 0; u < kMaxTreeBatch; ++u) {
                if (u < nb) {
                    const size_t base = (((size_t)b * p.N + js[u]) * p.Hkv + g) * D + lane * DPL;
                    load_slice<T, D>(kt + base, kf[u]);
                    load_slice<T, D>(vt + base, vf[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < kMaxTreeBatch; ++u) {
                if (u >= nb) continue;
                float dot = 0.f;
#pragma unroll
                for (int x = 0; x < DPL; ++x) dot = fmaf(qf[x], kf[u][x], dot);
                const float sc = warp_sum(dot) * L.scale_log2;
                const float mn = fmaxf(m_t, sc);
                const float alpha = exp2f(m_t - mn), pj = exp2f(sc - mn);
                l_t = l_t * alpha + pj;
#pragma unroll
                for (int x = 0; x < DPL; ++x) o[x] = fmaf(o[x], alpha, pj * vf[u][x]);
                m_t = mn;
            }
        }
    }

    // ---- committed prefix: partials of every CTA that covered this segment
    // (this kernel is launched as a programmatic dependent of the prefix
    // kernel: everything above overlaps its tail, nothing below may)
    //
    // The reads above (q, anc_mask, tree K/V), those of ctx_len just below
    // (which CTAs' partials cover this segment) and the status ORs come
    // before this kernel's own wait.  They are safe by transitivity: the
    // prefix kernel triggers its dependents only after its own pdl_wait() has
    // returned, i.e. after every kernel before it on the stream (the one that
    // wrote the masks, the caller's uploads) has completed and flushed.  So
    // once any block of this kernel runs, those inputs are final.  This holds
    // only while the prefix kernel keeps pdl_trigger() after pdl_wait().
    const int Lb = seq_len(a.ctx_len, b, p.max_pages, (i == 0 && h == 0 && gt == 0) ? a.status : nullptr);
    int count = 0, c_lo = 0;
    long long nT = 0;
    if (Lb > 0) {
        nT = total_tiles(p, a.ctx_len);
        const long long first = segment_offset(p, a.ctx_len, s);
        const long long last = first + tiles_of(Lb) - 1;
        c_lo = cta_of_tile(first, nT, p.Cg);
        count = cta_of_tile(last, nT, p.Cg) - c_lo + 1;
    }
    pdl_wait();
    const size_t sf = slot_floats(p);
    const float* ws = L.ws + slot_index(p, rg, c_lo, s) * sf;
    // with fewer tiles than CTAs some CTAs own no tile and write no partial
    const bool every_cta_owns = nT >= p.Cg;
    auto has_partial = [&](int k) {
        return k < count &&
               (every_cta_owns || cta_begin(c_lo + k, nT, p.Cg) != cta_begin(c_lo + k + 1, nT, p.Cg));
    };

    // Each warp folds partials w, w + W, w + 2 W, ... into its own running
    // (max, sum, output slice), which starts from its share of the tree block.
    // All of a round's loads (up to kR partials per warp: maxima, sums and
    // the row slices) are issued before any is used, so a round costs one trip
    // to L2.
    float m_w = m_t, l_w = l_t;
    for (int k0 = warp; k0 < count; k0 += W * kR) {
        float mk[kR], lk[kR];
        float part[kR][DPL];
#pragma unroll
        for (int u = 0; u < kR; ++u) {
            const int k = k0 + u * W;
            mk[u] = -INFINITY;
            lk[u] = 0.f;
            if (has_partial(k)) {
                const float* slot = ws + (size_t)k * sf;
                mk[u] = slot[(size_t)p.rg.RG * D + rl];
                lk[u] = slot[(size_t)p.rg.RG * D + p.rg.RG + rl];
                load_partial<DPL>(slot + (size_t)rl * D + lane * DPL, part[u]);
            } else {
#pragma unroll
                for (int x = 0; x < DPL; ++x) part[u][x] = 0.f;
            }
        }
        float mr = m_w;
#pragma unroll
        for (int u = 0; u < kR; ++u) mr = fmaxf(mr, mk[u]);
        if (mr > -INFINITY) {
            const float a0 = m_w > -INFINITY ? exp2f(m_w - mr) : 0.f;
            l_w *= a0;
#pragma unroll
            for (int x = 0; x < DPL; ++x) o[x] *= a0;
#pragma unroll
            for (int u = 0; u < kR; ++u) {
                const float w = mk[u] > -INFINITY ? exp2f(mk[u] - mr) : 0.f;
                l_w = fmaf(w, lk[u], l_w);
#pragma unroll
                for (int x = 0; x < DPL; ++x) o[x] = fmaf(part[u][x], w, o[x]);
            }
            m_w = mr;
        }
    }

    // ---- the warps' parts on the common shift
    if (lane == 0) s_red[warp] = m_w;
    group_sync(bar_id, 32 * W);
    float mmax = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) mmax = fmaxf(mmax, s_red[w]);
    const float aw = m_w > -INFINITY ? exp2f(m_w - mmax) : 0.f;
#pragma unroll
    for (int x = 0; x < DPL; ++x) s_o[warp][lane * DPL + x] = o[x] * aw;
    const float lsum = l_w * aw;  // the same in every lane of the warp
    group_sync(bar_id, 32 * W);   // every warp has read the maxima in s_red
    if (lane == 0) s_red[warp] = lsum;
    group_sync(bar_id, 32 * W);

    // ---- combine the warps' sums and write the row
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) l += s_red[w];
    const float inv = 1.f / l;
    float* orow = a.out + (size_t)row * D;
    for (int d = gt; d < D; d += 32 * W) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) v += s_o[w][d];
        v *= inv;
        orow[d] = v;
        if (!isfinite(v)) atomicOr(a.status, LUCETREE_DEV_NONFINITE);
    }
    if (a.lse && gt == 0) a.lse[row] = (mmax + log2f(l)) * kLn2;
}

}  // namespace merge

}  // namespace lucetree
