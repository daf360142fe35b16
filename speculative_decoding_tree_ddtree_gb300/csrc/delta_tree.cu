// delta_tree.cu -- tree-aware recurrent-state step of a gated-delta-rule
// (DeltaNet-style) layer, and its commit along the accepted path.
//
// Per value head the state S is [dk][dv] (fp32) and a tree node i with
// parent p (p = -1: the committed state S_root) gives
//     S_i = alpha_i (I - beta_i k_i k_i^T) S_p + beta_i k_i v_i^T,
//     o_i = S_i^T q_i.
// Column j of S only ever mixes with column j, so a CTA owns C columns of one
// (sequence, value head) and keeps that slice of every node's state in shared
// memory ([node][C][dk], column-major so a lane's four rows are one 16-byte
// load).  With u = k^T S_p and w = q^T S_p (one warp reduction for both),
//     d_j = beta (v_j - alpha u_j),   o_j = alpha w_j + (q . k) d_j,
//     S_i[r][j] = alpha S_p[r][j] + k_r d_j.
// Nodes are processed level by level (all nodes of one depth in parallel,
// one warp per node; a level only reads states of the level above), so the
// chain is the tree's depth, not its size.  Everything a level reads
// (q, k, the v slice, alpha, beta) is staged in shared memory by the prologue.
//
// The commit replays the accepted path (acc_nodes[b][0 .. acc_len[b])) from
// the committed state, one warp per (sequence, head, C columns) with the slice
// in registers, and writes the state back in place: rejected nodes never touch
// it.  dk = 128 (lane l owns rows 4l .. 4l+3).
#include "internal.cuh"
#include "delta.h"

namespace lucetree {

namespace {

constexpr int kDk = 128;
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

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

template <int C>
struct TreeSmem {
    static constexpr size_t bytes(int N) {
        return (size_t)(N + 1) * C * kDk * 4      // states: N nodes + the committed one
               + (size_t)2 * N * kDk * 4          // q, k (fp32)
               + (size_t)N * C * 4                // v slice
               + (size_t)2 * N * 4                // alpha, beta
               + (size_t)4 * 64 * 4 + 16;         // parent, order, level starts, flags
    }
};

template <bool BF16, int C>
__global__ void __launch_bounds__(kThreads) delta_tree_kernel(lucetree_delta_args a) {
    extern __shared__ __align__(16) float sm[];
    const int N = a.N, Hv = a.Hv, Hk = a.Hk, dv = a.dv;
    const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hk = h / (Hv / Hk), c0 = slice * C;
    float* st = sm;                                    // [N + 1][C][kDk]; slot N = committed state
    float* sq = st + (size_t)(N + 1) * C * kDk;        // [N][kDk]
    float* sk = sq + (size_t)N * kDk;                  // [N][kDk]
    float* sv = sk + (size_t)N * kDk;                  // [N][C]
    float* sal = sv + (size_t)N * C;                   // [N]
    float* sbe = sal + N;                              // [N]
    int* spar = reinterpret_cast<int*>(sbe + N);       // [64]
    int* sord = spar + 64;                             // [64] nodes by depth
    int* slvl = sord + 64;                             // [65] level starts
    int* sflag = slvl + 65;                            // [64] has children; [0..] reused
    __shared__ int n_levels;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();

    // ---- prologue: tree, inputs, committed state slice
    for (int i = threadIdx.x; i < N; i += kThreads) {
        int p = a.parent[(size_t)b * N + i];
        if (p < -1 || p >= i) {
            atomicOr(a.status, LUCETREE_DEV_BAD_PARENT);
            p = -1;
        }
        spar[i] = p;
        sflag[i] = 0;
    }
    {
        const uint16_t* q = reinterpret_cast<const uint16_t*>(a.q);
        const uint16_t* k = reinterpret_cast<const uint16_t*>(a.k);
        for (int e = threadIdx.x; e < N * kDk; e += kThreads) {
            const int i = e / kDk, r = e % kDk;
            const size_t off = (((size_t)b * N + i) * Hk + hk) * kDk + r;
            sq[e] = to_f32<BF16>(q[off]);
            sk[e] = to_f32<BF16>(k[off]);
        }
        const uint16_t* v = reinterpret_cast<const uint16_t*>(a.v);
        for (int e = threadIdx.x; e < N * C; e += kThreads) {
            const int i = e / C, j = e % C;
            sv[e] = to_f32<BF16>(v[(((size_t)b * N + i) * Hv + h) * dv + c0 + j]);
        }
        for (int i = threadIdx.x; i < N; i += kThreads) {
            sal[i] = a.alpha[((size_t)b * N + i) * Hv + h];
            sbe[i] = a.beta[((size_t)b * N + i) * Hv + h];
        }
        const float* s0 = a.state + ((size_t)b * Hv + h) * kDk * dv + c0;
        float* root = st + (size_t)N * C * kDk;
        for (int e = threadIdx.x; e < kDk * (C / 4); e += kThreads) {
            const int r = e / (C / 4), j4 = 4 * (e % (C / 4));
            const float4 x = *reinterpret_cast<const float4*>(s0 + (size_t)r * dv + j4);
            root[(j4 + 0) * kDk + r] = x.x;
            root[(j4 + 1) * kDk + r] = x.y;
            root[(j4 + 2) * kDk + r] = x.z;
            root[(j4 + 3) * kDk + r] = x.w;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // depth by parent (parents precede children), then a counting sort
        int depth[64], cnt[65];
        int maxd = 0;
        for (int d = 0; d <= N; ++d) cnt[d] = 0;
        for (int i = 0; i < N; ++i) {
            const int p = spar[i];
            depth[i] = p < 0 ? 0 : depth[p] + 1;
            if (p >= 0) sflag[p] = 1;
            maxd = max(maxd, depth[i]);
            ++cnt[depth[i]];
        }
        slvl[0] = 0;
        for (int d = 0; d <= maxd; ++d) slvl[d + 1] = slvl[d] + cnt[d];
        for (int d = 0; d <= maxd; ++d) cnt[d] = slvl[d];
        for (int i = 0; i < N; ++i) sord[cnt[depth[i]]++] = i;
        n_levels = maxd + 1;
    }
    __syncthreads();

    // ---- levels
    constexpr int V = 2 * C;
    constexpr int kGroup = 32 / V;  // lanes holding the same reduced value
    const int nl = n_levels;
    for (int lv = 0; lv < nl; ++lv) {
        for (int x = slvl[lv] + warp; x < slvl[lv + 1]; x += kWarps) {
            const int i = sord[x];
            const int p = spar[i];
            const float* sp = st + (size_t)(p < 0 ? N : p) * C * kDk;
            const float4 k4 = *reinterpret_cast<const float4*>(sk + (size_t)i * kDk + 4 * lane);
            const float4 q4 = *reinterpret_cast<const float4*>(sq + (size_t)i * kDk + 4 * lane);
            float part[V];
#pragma unroll
            for (int j = 0; j < C; ++j) {
                const float4 s4 = *reinterpret_cast<const float4*>(sp + (size_t)j * kDk + 4 * lane);
                part[j] = k4.x * s4.x + k4.y * s4.y + k4.z * s4.z + k4.w * s4.w;
                part[C + j] = q4.x * s4.x + q4.y * s4.y + q4.z * s4.z + q4.w * s4.w;
            }
            const float qk = warp_sum(q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w);
            const float red = reduce_scatter<V>(part, lane);      // u_j (idx < C) or w_{idx - C}
            const int idx = lane / kGroup;
            const float w = __shfl_sync(0xffffffffu, red, (lane + C * kGroup) & 31);
            const float al = sal[i], be = sbe[i];
            float d = 0.f;
            if (idx < C) {
                d = be * (sv[i * C + idx] - al * red);
                if (lane % kGroup == 0)
                    a.out[(((size_t)b * N + i) * Hv + h) * dv + c0 + idx] = al * w + qk * d;
            }
            if (sflag[i]) {
                float* si = st + (size_t)i * C * kDk;
#pragma unroll
                for (int j = 0; j < C; ++j) {
                    const float dj = __shfl_sync(0xffffffffu, d, j * kGroup);
                    const float4 s4 = *reinterpret_cast<const float4*>(sp + (size_t)j * kDk + 4 * lane);
                    float4 n4;
                    n4.x = fmaf(k4.x, dj, al * s4.x);
                    n4.y = fmaf(k4.y, dj, al * s4.y);
                    n4.z = fmaf(k4.z, dj, al * s4.z);
                    n4.w = fmaf(k4.w, dj, al * s4.w);
                    *reinterpret_cast<float4*>(si + (size_t)j * kDk + 4 * lane) = n4;
                }
            }
        }
        __syncthreads();
    }
}

// One warp per (slice, head, sequence); the state slice stays in registers.
template <bool BF16, int C>
__global__ void __launch_bounds__(32) delta_commit_kernel(lucetree_delta_args a) {
    const int N = a.N, Hv = a.Hv, Hk = a.Hk, dv = a.dv;
    const int slice = blockIdx.x, h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x;
    const int hk = h / (Hv / Hk), c0 = slice * C;
    pdl_wait();
    if (lane == 0) pdl_trigger();
    int n_acc = a.acc_len[b];
    if (n_acc < 0 || n_acc > N) {
        if (lane == 0 && slice == 0 && h == 0) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
        return;
    }
    if (n_acc == 0) return;  // nothing accepted: the committed state stays as it is
    float* s0 = a.state + ((size_t)b * Hv + h) * kDk * dv + c0;
    float S[4][C];
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j4 = 0; j4 < C; j4 += 4) {
            const float4 x = *reinterpret_cast<const float4*>(s0 + (size_t)(4 * lane + m) * dv + j4);
            S[m][j4] = x.x;
            S[m][j4 + 1] = x.y;
            S[m][j4 + 2] = x.z;
            S[m][j4 + 3] = x.w;
        }
    const uint16_t* kp = reinterpret_cast<const uint16_t*>(a.k);
    const uint16_t* vp = reinterpret_cast<const uint16_t*>(a.v);
    constexpr int kGroup = 32 / C;
    for (int t = 0; t < n_acc; ++t) {
        const int i = a.acc_nodes[(size_t)b * N + t];
        if (i < 0 || i >= N) {
            if (lane == 0 && slice == 0 && h == 0) atomicOr(a.status, LUCETREE_DEV_BAD_NODE);
            return;  // the state is left as it was
        }
        const size_t node = (size_t)b * N + i;
        const uint2 kb = *reinterpret_cast<const uint2*>(kp + (node * Hk + hk) * kDk + 4 * lane);
        const float kr[4] = {to_f32<BF16>((uint16_t)(kb.x & 0xFFFFu)), to_f32<BF16>((uint16_t)(kb.x >> 16)),
                             to_f32<BF16>((uint16_t)(kb.y & 0xFFFFu)), to_f32<BF16>((uint16_t)(kb.y >> 16))};
        float part[C];
#pragma unroll
        for (int j = 0; j < C; ++j) part[j] = kr[0] * S[0][j] + kr[1] * S[1][j] + kr[2] * S[2][j] + kr[3] * S[3][j];
        const float u = reduce_scatter<C>(part, lane);  // u_{lane / kGroup}
        const float al = a.alpha[node * Hv + h], be = a.beta[node * Hv + h];
        const float d = be * (to_f32<BF16>(vp[(node * Hv + h) * dv + c0 + lane / kGroup]) - al * u);
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float dj = __shfl_sync(0xffffffffu, d, j * kGroup);
#pragma unroll
            for (int m = 0; m < 4; ++m) S[m][j] = fmaf(kr[m], dj, al * S[m][j]);
        }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int j4 = 0; j4 < C; j4 += 4)
            *reinterpret_cast<float4*>(s0 + (size_t)(4 * lane + m) * dv + j4) =
                make_float4(S[m][j4], S[m][j4 + 1], S[m][j4 + 2], S[m][j4 + 3]);
}

template <bool BF16, int C>
cudaError_t launch_tree_c(const lucetree_delta_args& a, cudaStream_t stream) {
    auto kern = delta_tree_kernel<BF16, C>;
    const size_t smem = TreeSmem<C>::bytes(a.N);
    static size_t configured = 0;  // largest dynamic shared memory size set so far
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    return launch_pdl(kern, dim3(a.dv / C, a.Hv, a.B), dim3(kThreads), smem, stream, a);
}

}  // namespace

int delta_tree_columns(int N) { return N <= 26 ? 8 : 4; }

size_t delta_tree_smem_bytes(int N) {
    return delta_tree_columns(N) == 8 ? TreeSmem<8>::bytes(N) : TreeSmem<4>::bytes(N);
}

cudaError_t launch_delta_tree(const lucetree_delta_args& a, cudaStream_t stream) {
    const bool bf = a.dtype == LUCETREE_BF16;
    if (delta_tree_columns(a.N) == 8) return bf ? launch_tree_c<true, 8>(a, stream) : launch_tree_c<false, 8>(a, stream);
    return bf ? launch_tree_c<true, 4>(a, stream) : launch_tree_c<false, 4>(a, stream);
}

cudaError_t launch_delta_commit(const lucetree_delta_args& a, cudaStream_t stream) {
    constexpr int C = 8;
    const dim3 grid(a.dv / C, a.Hv, a.B);
    if (a.dtype == LUCETREE_BF16) return launch_pdl(delta_commit_kernel<true, C>, grid, dim3(32), 0, stream, a);
    return launch_pdl(delta_commit_kernel<false, C>, grid, dim3(32), 0, stream, a);
}

}  // namespace lucetree
