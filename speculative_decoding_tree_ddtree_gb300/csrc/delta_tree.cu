// delta_tree.cu -- tree-aware recurrent-state step of a gated-delta-rule
// (DeltaNet-style) layer, and its commit along the accepted path.
//
// Per value head the state S is [dk][dv] (fp32) and a tree node i with
// parent p (p = -1: the committed state S_root) gives
//     S_i = alpha_i (I - beta_i k_i k_i^T) S_p + beta_i k_i v_i^T,
//     o_i = S_i^T q_i.
// Column j of S only ever mixes with column j, so a CTA owns C = 8 columns of
// one (sequence, value head).  With u = k^T S_p and w = q^T S_p (one warp
// reduction for both),
//     d_j = beta (v_j - alpha u_j),   o_j = alpha w_j + (q . k) d_j,
//     S_i[r][j] = alpha S_p[r][j] + k_r d_j.
//
// Tree pass: every node lies on the root path of some leaf, so each warp
// takes leaves in turn and replays the leaf's root path from the committed
// state with the state slice in registers (lane l owns rows 4l .. 4l+3),
// writing every node's output on the way.  A node on the paths of several
// leaves is recomputed by the same instruction sequence from the same inputs,
// so the repeated writes carry identical values.  Nothing but inputs lives in
// shared memory (q, k, the v slice, the gates, staged once), so every CTA of
// a head fits on the chip at once; the cost is the sum of the leaves' depths
// per CTA, and a chain is a single replay.
//
// The commit replays the accepted path (acc_nodes[b][0 .. acc_len[b])) the
// same way and writes the state back in place: rejected nodes never touch it.
// dk = 128.
#include "internal.cuh"
#include "delta.h"

namespace lucetree {

namespace {

constexpr int kDk = 128;
constexpr int kC = 8;                 // state columns per CTA
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxN = 64;

// Sum of each of V values over the warp's 32 lanes, scattered: recursive
// halving over the top log2(V) lane bits, then a butterfly over the rest.
// Lane l returns the sum of value l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane) {
    constexpr int L = V == 8 ? 3 : (V == 16 ? 4 : 5);
#pragma unroll
    for (int s = 0; s < L; ++s) {
        const int m = 16 >> s;
        const int n = V >> (s + 1);
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = upper ? v[i] : v[i + n];
            const float keep = upper ? v[i + n] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
#pragma unroll
    for (int s = L; s < 5; ++s) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> s);
    return v[0];
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t b) {
    if constexpr (BF16) return __uint_as_float((uint32_t)b << 16);
    else return __half2float(__ushort_as_half(b));
}

template <bool BF16>
__device__ __forceinline__ float4 load4(const uint16_t* p) {  // four 16-bit values, 8-byte aligned
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    return make_float4(to_f32<BF16>((uint16_t)(x.x & 0xFFFFu)), to_f32<BF16>((uint16_t)(x.x >> 16)),
                       to_f32<BF16>((uint16_t)(x.y & 0xFFFFu)), to_f32<BF16>((uint16_t)(x.y >> 16)));
}

// Staged inputs of one CTA: per node the key (and query) rows, the CTA's v
// columns, the gates and q . k.
struct Stage {
    float* k;     // [N][kDk]
    float* q;     // [N][kDk] (tree pass only)
    float* v;     // [N][vs], this warp's first column at v[0]
    int vs;       // row stride of v
    float* al;    // [N]
    float* be;    // [N]
    float* qk;    // [N] (tree pass only)
};

// dynamic shared memory: k (and q) rows, ncol v columns, the gates (and q . k)
__host__ __device__ constexpr size_t stage_bytes(int N, bool with_q, int ncol) {
    return (size_t)N * kDk * 4 * (with_q ? 2 : 1) + (size_t)N * (ncol + (with_q ? 3 : 2)) * 4;
}

// One node of the recurrence on the warp's register state S[m][j] = S[4l+m][c0+j].
// With EMIT, also returns the node's output column (on lanes 4j, j < 8).
template <bool EMIT>
__device__ __forceinline__ float delta_step(float (&S)[4][kC], const Stage& sg, int n, int lane) {
    const float4 k4 = *reinterpret_cast<const float4*>(sg.k + (size_t)n * kDk + 4 * lane);
    const float kr[4] = {k4.x, k4.y, k4.z, k4.w};
    constexpr int V = EMIT ? 2 * kC : kC;
    float part[V];
#pragma unroll
    for (int j = 0; j < kC; ++j) part[j] = kr[0] * S[0][j] + kr[1] * S[1][j] + kr[2] * S[2][j] + kr[3] * S[3][j];
    if constexpr (EMIT) {
        const float4 q4 = *reinterpret_cast<const float4*>(sg.q + (size_t)n * kDk + 4 * lane);
#pragma unroll
        for (int j = 0; j < kC; ++j)
            part[kC + j] = q4.x * S[0][j] + q4.y * S[1][j] + q4.z * S[2][j] + q4.w * S[3][j];
    }
    constexpr int kGroup = 32 / V;
    const float red = reduce_scatter<V>(part, lane);  // u_{lane / kGroup} (or w_{lane / kGroup - kC})
    const int idx = lane / kGroup;
    const float al = sg.al[n], be = sg.be[n];
    float d = 0.f, o = 0.f;
    if (idx < kC) d = be * (sg.v[n * sg.vs + idx] - al * red);
    if constexpr (EMIT) {
        const float w = __shfl_sync(0xffffffffu, red, (lane + kC * kGroup) & 31);
        o = al * w + sg.qk[n] * d;
    }
#pragma unroll
    for (int j = 0; j < kC; ++j) {
        const float dj = __shfl_sync(0xffffffffu, d, j * kGroup);
#pragma unroll
        for (int m = 0; m < 4; ++m) S[m][j] = fmaf(kr[m], dj, al * S[m][j]);
    }
    return o;
}

__device__ __forceinline__ void load_state(float (&S)[4][kC], const float* s0, int dv, int lane) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j4 = 0; j4 < kC; j4 += 4) {
            const float4 x = *reinterpret_cast<const float4*>(s0 + (size_t)(4 * lane + m) * dv + j4);
            S[m][j4] = x.x;
            S[m][j4 + 1] = x.y;
            S[m][j4 + 2] = x.z;
            S[m][j4 + 3] = x.w;
        }
}

// Stage the inputs of nodes list[0 .. n) (list = nullptr: nodes 0 .. n) into
// sg: k (and q) rows, v columns c0 .. c0 + sg.vs (those below dv), the gates.
// Each thread issues kB loads before it stores any, so the staging costs one
// or two memory round trips rather than one per element group.
template <bool BF16, bool WITH_Q>
__device__ void stage_inputs(const lucetree_delta_args& a, const Stage& sg, const int* list, int n, int b, int h,
                             int hk, int c0) {
    constexpr int kB = 8;
    const uint16_t* kp = reinterpret_cast<const uint16_t*>(a.k);
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(a.q);
    const uint16_t* vp = reinterpret_cast<const uint16_t*>(a.v);
    const int total = n * (kDk / 4);
    for (int e0 = threadIdx.x; e0 < total; e0 += kB * kThreads) {
        uint2 xk[kB], xq[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) {
                const int t = e / (kDk / 4), r = 4 * (e % (kDk / 4));
                const size_t off = (((size_t)b * a.N + (list ? list[t] : t)) * a.Hk + hk) * kDk + r;
                xk[u] = *reinterpret_cast<const uint2*>(kp + off);
                if constexpr (WITH_Q) xq[u] = *reinterpret_cast<const uint2*>(qp + off);
            }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
            const int e = e0 + u * kThreads;
            if (e < total) {
                const int t = e / (kDk / 4), r = 4 * (e % (kDk / 4));
                auto cvt = [](uint2 x) {
                    return make_float4(to_f32<BF16>((uint16_t)(x.x & 0xFFFFu)), to_f32<BF16>((uint16_t)(x.x >> 16)),
                                       to_f32<BF16>((uint16_t)(x.y & 0xFFFFu)), to_f32<BF16>((uint16_t)(x.y >> 16)));
                };
                *reinterpret_cast<float4*>(sg.k + (size_t)t * kDk + r) = cvt(xk[u]);
                if constexpr (WITH_Q) *reinterpret_cast<float4*>(sg.q + (size_t)t * kDk + r) = cvt(xq[u]);
            }
        }
    }
    const int tv = n * sg.vs;
    for (int e0 = threadIdx.x; e0 < tv + 2 * n; e0 += 4 * kThreads) {
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            x[u] = 0.f;
            if (e < tv) {
                const int t = e / sg.vs, j = e % sg.vs;
                if (c0 + j < a.dv)
                    x[u] = to_f32<BF16>(vp[(((size_t)b * a.N + (list ? list[t] : t)) * a.Hv + h) * a.dv + c0 + j]);
            } else if (e < tv + 2 * n) {
                const int t = (e - tv) >> 1;
                const size_t g = ((size_t)b * a.N + (list ? list[t] : t)) * a.Hv + h;
                x[u] = ((e - tv) & 1) ? a.beta[g] : a.alpha[g];
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * kThreads;
            if (e < tv) sg.v[e] = x[u];
            else if (e < tv + 2 * n) (((e - tv) & 1) ? sg.be : sg.al)[(e - tv) >> 1] = x[u];
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) delta_tree_kernel(lucetree_delta_args a) {
    extern __shared__ __align__(16) float sm[];
    __shared__ int spar[kMaxN], sleaf[kMaxN], schild[kMaxN], spath[kWarps][kMaxN], splen[kWarps];
    __shared__ __align__(16) float sroot[kC * kDk];  // committed state slice, [column][row]
    __shared__ int n_leaves;
    const int N = a.N, Hv = a.Hv, dv = a.dv;
    const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / (Hv / a.Hk), c0 = slice * kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Stage sg;
    sg.k = sm;
    sg.q = sg.k + (size_t)N * kDk;
    sg.v = sg.q + (size_t)N * kDk;
    sg.vs = kC;
    sg.al = sg.v + (size_t)N * kC;
    sg.be = sg.al + N;
    sg.qk = sg.be + N;

    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();

    // ---- tree (invalid parents become root children), committed slice, inputs
    const float* s0 = a.state + ((size_t)b * Hv + h) * kDk * dv + c0;
    {
        // kDk rows x kC columns: two 16-byte loads per thread, stored column-major
        float4 x[kC * kDk / 4 / kThreads];
#pragma unroll
        for (int u = 0; u < kC * kDk / 4 / kThreads; ++u) {
            const int e = threadIdx.x + u * kThreads, r = e / (kC / 4), j4 = 4 * (e % (kC / 4));
            x[u] = *reinterpret_cast<const float4*>(s0 + (size_t)r * dv + j4);
        }
        for (int i = threadIdx.x; i < N; i += kThreads) {
            int p = a.parent[(size_t)b * N + i];
            if (p < -1 || p >= i) {
                atomicOr(a.status, LUCETREE_DEV_BAD_PARENT);
                p = -1;
            }
            spar[i] = p;
            schild[i] = 0;
        }
#pragma unroll
        for (int u = 0; u < kC * kDk / 4 / kThreads; ++u) {
            const int e = threadIdx.x + u * kThreads, r = e / (kC / 4), j4 = 4 * (e % (kC / 4));
            sroot[(j4 + 0) * kDk + r] = x[u].x;
            sroot[(j4 + 1) * kDk + r] = x[u].y;
            sroot[(j4 + 2) * kDk + r] = x[u].z;
            sroot[(j4 + 3) * kDk + r] = x[u].w;
        }
    }
    stage_inputs<BF16, true>(a, sg, nullptr, N, b, h, hk, c0);
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += kThreads)
        if (spar[i] >= 0) schild[spar[i]] = 1;
    __syncthreads();
    if (warp == 0) {
        int cnt = 0;
        for (int base = 0; base < N; base += 32) {
            const int i = base + lane;
            const bool leaf = i < N && !schild[i];
            const unsigned m = __ballot_sync(0xffffffffu, leaf);
            if (leaf) sleaf[cnt + __popc(m & ((1u << lane) - 1u))] = i;
            cnt += __popc(m);
        }
        if (lane == 0) n_leaves = cnt;
    }
    for (int i = warp; i < N; i += kWarps) {
        const float4 q4 = *reinterpret_cast<const float4*>(sg.q + (size_t)i * kDk + 4 * lane);
        const float4 k4 = *reinterpret_cast<const float4*>(sg.k + (size_t)i * kDk + 4 * lane);
        const float qk = warp_sum(q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w);
        if (lane == 0) sg.qk[i] = qk;
    }
    __syncthreads();

    // ---- one leaf's root path per warp at a time
    int* path = spath[warp];
    for (int x = warp; x < n_leaves; x += kWarps) {
        if (lane == 0) {
            int len = 0;
            for (int j = sleaf[x]; j >= 0 && len < kMaxN; j = spar[j]) path[len++] = j;  // leaf first
            splen[warp] = len;
        }
        __syncwarp();
        float S[4][kC];
#pragma unroll
        for (int j = 0; j < kC; ++j) {
            const float4 x4 = *reinterpret_cast<const float4*>(sroot + j * kDk + 4 * lane);
            S[0][j] = x4.x;
            S[1][j] = x4.y;
            S[2][j] = x4.z;
            S[3][j] = x4.w;
        }
        for (int t = splen[warp] - 1; t >= 0; --t) {
            const int n = path[t];
            const float o = delta_step<true>(S, sg, n, lane);
            if ((lane & 1) == 0 && lane < 2 * kC) a.out[(((size_t)b * N + n) * Hv + h) * dv + c0 + (lane >> 1)] = o;
        }
        __syncwarp();
    }
}

// The commit: a CTA covers kWarps column slices of one (sequence, head),
// stages the accepted path's inputs once, and each warp replays the path on
// its slice in registers and writes it back.
template <bool BF16>
__global__ void __launch_bounds__(kThreads) delta_commit_kernel(lucetree_delta_args a) {
    extern __shared__ __align__(16) float sm[];
    __shared__ int snode[kMaxN];
    __shared__ int s_bad;
    const int N = a.N, Hv = a.Hv, dv = a.dv;
    const int h = blockIdx.y, b = blockIdx.z;
    const int hk = h / (Hv / a.Hk), cb = blockIdx.x * kWarps * kC;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool report = blockIdx.x == 0 && h == 0 && threadIdx.x == 0;
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    // the state slice first: its loads overlap the path's
    const int c0 = cb + warp * kC;
    float* s0 = a.state + ((size_t)b * Hv + h) * kDk * dv + (c0 < dv ? c0 : 0);
    float S[4][kC];
    load_state(S, s0, dv, lane);
    const int n_acc = a.acc_len[b];
    if (n_acc < 0 || n_acc > N) {
        if (report) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
        return;
    }
    if (n_acc == 0) return;  // nothing accepted: the committed state stays as it is
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < n_acc; t += kThreads) {
        const int i = a.acc_nodes[(size_t)b * N + t];
        const bool ok = i >= 0 && i < N;
        if (!ok) s_bad = 1;
        snode[t] = ok ? i : 0;
    }
    __syncthreads();
    if (s_bad) {  // uniform: leave this sequence's state as it was
        if (report) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
        return;
    }
    Stage sg;
    sg.k = sm;
    sg.q = nullptr;
    sg.v = sg.k + (size_t)N * kDk;
    sg.vs = kWarps * kC;
    sg.al = sg.v + (size_t)N * kWarps * kC;
    sg.be = sg.al + N;
    sg.qk = nullptr;
    stage_inputs<BF16, false>(a, sg, snode, n_acc, b, h, hk, cb);
    __syncthreads();
    if (c0 >= dv) return;
    Stage mine = sg;
    mine.v = sg.v + warp * kC;
    for (int t = 0; t < n_acc; ++t) delta_step<false>(S, mine, t, lane);
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j4 = 0; j4 < kC; j4 += 4)
            *reinterpret_cast<float4*>(s0 + (size_t)(4 * lane + m) * dv + j4) =
                make_float4(S[m][j4], S[m][j4 + 1], S[m][j4 + 2], S[m][j4 + 3]);
}

template <bool BF16>
cudaError_t launch_tree_t(const lucetree_delta_args& a, cudaStream_t stream) {
    // the limit is raised to the largest tree the kernel takes (64 nodes), so
    // launches of different sizes from several threads never lower it
    static SmemLimitSeen seen;
    const size_t smem = delta_tree_smem_bytes(a.N);
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(delta_tree_kernel<BF16>),
                                     (int)delta_tree_smem_bytes(64), seen);
    if (e != cudaSuccess) return e;
    return launch_pdl(delta_tree_kernel<BF16>, dim3(a.dv / kC, a.Hv, a.B), dim3(kThreads), smem, stream, a);
}

template <bool BF16>
cudaError_t launch_commit_t(const lucetree_delta_args& a, cudaStream_t stream) {
    static SmemLimitSeen seen;
    const size_t smem = stage_bytes(a.N, false, kWarps * kC);
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(delta_commit_kernel<BF16>),
                                     (int)stage_bytes(64, false, kWarps * kC), seen);
    if (e != cudaSuccess) return e;
    const int per_cta = kWarps * kC;
    return launch_pdl(delta_commit_kernel<BF16>, dim3((a.dv + per_cta - 1) / per_cta, a.Hv, a.B), dim3(kThreads),
                      smem, stream, a);
}

}  // namespace

size_t delta_tree_smem_bytes(int N) { return stage_bytes(N, true, kC); }

cudaError_t launch_delta_tree(const lucetree_delta_args& a, cudaStream_t stream) {
    return a.dtype == LUCETREE_BF16 ? launch_tree_t<true>(a, stream) : launch_tree_t<false>(a, stream);
}

cudaError_t launch_delta_commit(const lucetree_delta_args& a, cudaStream_t stream) {
    return a.dtype == LUCETREE_BF16 ? launch_commit_t<true>(a, stream) : launch_commit_t<false>(a, stream);
}

}  // namespace lucetree
