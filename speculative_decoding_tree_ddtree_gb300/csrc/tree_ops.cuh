// tree_ops.cuh -- greedy acceptance and the commit copy as warp / CTA device
// routines, shared by their own kernels and by the fused verify step.
//
// Acceptance follows the greedy (temperature 0) rule: a draft node is right
// when its token equals the argmax of its parent's logits, and the step keeps
// the longest root path of right nodes (PyTorch Korea forum post "Lucebox:
// 추측 디코딩과 전용 커널로 ...", section "Lucebox 설치 및 실행").  Commit copies
// the kept nodes' K/V into the 64-token pages after the committed prefix and
// leaves rejected nodes unwritten, which is the KV rollback of the
// DFlashTarget interface ("Lucebox Hub", section "Speculative decoding 계층").
#pragma once

#include "internal.cuh"

namespace lucetree {
namespace tree {

// Ancestor-or-self mask of node i by walking par[] (a row of N parents,
// typically in shared memory) up to the root: bit i, then every ancestor.
// A parent outside [-1, c) stops the walk and sets *bad.
__device__ inline uint64_t anc_walk(const int32_t* par, int i, bool* bad) {
    uint64_t m = 1ull << i;
    int c = i;
    for (int guard = 0; guard < LUCETREE_MAX_NODES; ++guard) {
        const int p = par[c];
        if (p == -1) return m;
        if (p < -1 || p >= c) {
            *bad = true;
            return m;
        }
        m |= 1ull << p;
        c = p;
    }
    return m;
}

// One warp decides sequence b.  Lanes load the tree (node i in lane i % 32)
// and decide whether each node's draft token equals its parent row's argmax;
// the ok-flags (node and all ancestors match) and depths then follow in node
// order.  The deepest ok node (lowest id among equals: ids are scanned upward
// with a strict comparison) ends the accepted path.  `am` (the argmax rows
// [N + 1] of this sequence) is read through L2, so it may have been written
// by another CTA of the same grid that fenced before signalling.
__device__ inline void accept_warp(const int32_t* __restrict__ par, const int32_t* __restrict__ dr,
                                   const int32_t* am, int N, int vocab, int32_t* __restrict__ out,
                                   int32_t* __restrict__ acc_len_b, int32_t* __restrict__ bonus_b,
                                   uint32_t* status) {
    const int lane = threadIdx.x & 31;
    int p[2] = {-1, -1};
    bool match[2] = {false, false};
    bool bad = false, bad_tok = false;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int i = lane + 32 * k;
        if (i < N) {
            p[k] = par[i];
            if (p[k] < -1 || p[k] >= i) {
                bad = true;
            } else {
                const int t = dr[i];
                if (t < 0 || t >= vocab) bad_tok = true;
                else match[k] = t == __ldcg(am + p[k] + 1);
            }
        }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (__any_sync(0xffffffffu, bad_tok) && lane == 0) atomicOr(status, LUCETREE_DEV_BAD_TOKEN);
    const uint32_t mlo = __ballot_sync(0xffffffffu, match[0]), mhi = __ballot_sync(0xffffffffu, match[1]);
    const uint64_t matched = ((uint64_t)mhi << 32) | mlo;
    int best = -1, best_depth = 0;
    uint64_t ok = 0;
    int d0 = 0, d1 = 0;  // depths of this lane's nodes
    if (!bad) {
        for (int i = 0; i < N; ++i) {
            const int pi = __shfl_sync(0xffffffffu, i < 32 ? p[0] : p[1], i & 31);
            int dp = 0;
            if (pi >= 0) {
                const int a0 = __shfl_sync(0xffffffffu, d0, pi & 31), a1 = __shfl_sync(0xffffffffu, d1, pi & 31);
                dp = pi < 32 ? a0 : a1;
            }
            const int di = dp + 1;
            if ((i & 31) == lane) {
                if (i < 32) d0 = di;
                else d1 = di;
            }
            const bool ok_i = ((matched >> i) & 1ull) && (pi < 0 || ((ok >> pi) & 1ull));
            if (ok_i) {
                ok |= 1ull << i;
                if (di > best_depth) {
                    best = i;
                    best_depth = di;
                }
            }
        }
    } else if (lane == 0) {
        atomicOr(status, LUCETREE_DEV_BAD_PARENT);
    }
    for (int k = best_depth + lane; k < N; k += 32) out[k] = -1;
    if (lane == 0) {
        int k = best_depth;
        for (int c = best; c >= 0; c = par[c]) out[--k] = c;
        *acc_len_b = best_depth;
        *bonus_b = __ldcg(am + best + 1);
    }
}

// The whole CTA commits sequence b: 16-byte copies of every accepted node's K
// and V rows (all KV heads).  The length is written after the CTA has read
// ctx_len_in, so ctx_len_out may alias it.  acc_nodes / acc_len are read
// through L2 (they may come from another warp or CTA that fenced first).
// s_good: one shared int.
__device__ inline void commit_block(const lucetree_commit_args& c, int b, int elem_bytes, int* s_good) {
    const int L = c.ctx_len_in[b];
    const int a = __ldcg(c.acc_len + b);
    if (threadIdx.x == 0) *s_good = 0x7fffffff;
    __syncthreads();
    const size_t row_bytes = (size_t)c.D * elem_bytes;
    const int vec_per_row = (int)(row_bytes / 16);
    const char* kt = reinterpret_cast<const char*>(c.k_tree);
    const char* vt = reinterpret_cast<const char*>(c.v_tree);
    char* kp = reinterpret_cast<char*>(c.k_pool);
    char* vp = reinterpret_cast<char*>(c.v_pool);
    int count = a;
    if (a < 0 || a > c.N || L < 0) {
        if (threadIdx.x == 0) atomicOr(c.status, a < 0 || a > c.N ? LUCETREE_DEV_BAD_NODE : LUCETREE_DEV_BAD_CTX);
        count = 0;
    }
    // validate entries first so the copy stops at the first bad one
    for (int k = threadIdx.x; k < count; k += blockDim.x) {
        const int node = __ldcg(c.acc_nodes + (size_t)b * c.N + k);
        const long long pos = (long long)L + k;
        const long long pi = pos / kPage;
        bool good = node >= 0 && node < c.N && pi < c.max_pages_per_seq;
        uint32_t flag = (node >= 0 && node < c.N) ? LUCETREE_DEV_BAD_PAGE : LUCETREE_DEV_BAD_NODE;
        if (good) {
            const int page = c.page_table[(size_t)b * c.max_pages_per_seq + pi];
            good = page >= 0 && page < c.num_pages;
        }
        if (!good) {
            atomicOr(c.status, flag);
            atomicMin(s_good, k);
        }
    }
    __syncthreads();
    count = min(count, *s_good);
    const int units = count * c.Hkv * vec_per_row;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        const int v = u % vec_per_row;
        const int g = (u / vec_per_row) % c.Hkv;
        const int k = u / (vec_per_row * c.Hkv);
        const int node = __ldcg(c.acc_nodes + (size_t)b * c.N + k);
        const long long pos = (long long)L + k;
        const int page = c.page_table[(size_t)b * c.max_pages_per_seq + pos / kPage];
        const size_t dst = ((((size_t)page * c.Hkv + g) * kPage + (size_t)(pos % kPage)) * row_bytes) + (size_t)v * 16;
        const size_t src = ((((size_t)b * c.N + node) * c.Hkv + g) * row_bytes) + (size_t)v * 16;
        *reinterpret_cast<uint4*>(kp + dst) = *reinterpret_cast<const uint4*>(kt + src);
        *reinterpret_cast<uint4*>(vp + dst) = *reinterpret_cast<const uint4*>(vt + src);
    }
    __syncthreads();
    if (threadIdx.x == 0) c.ctx_len_out[b] = L < 0 ? L : L + count;
}

}  // namespace tree
}  // namespace lucetree
