// tree_ops.cu -- ancestor masks, greedy acceptance and the commit copy.
//
// Acceptance follows the greedy (temperature 0) rule: a draft node is right
// when its token equals the argmax of its parent's logits, and the step keeps
// the longest root path of right nodes (PyTorch Korea forum post "Lucebox:
// 추측 디코딩과 전용 커널로 ...", section "Lucebox 설치 및 실행").  Commit copies
// the kept nodes' K/V into the 64-token pages after the committed prefix and
// leaves rejected nodes unwritten, which is the KV rollback of the
// DFlashTarget interface ("Lucebox Hub", section "Speculative decoding 계층").
#include "internal.cuh"

namespace lucetree {

namespace {

// One warp per sequence; node i lives in lane i % 32, slot i / 32.  Parents
// are loaded in parallel, then the masks are built in node order (each node
// needs its parent's mask) with shuffles instead of dependent global loads.
__global__ void __launch_bounds__(128) build_anc_kernel(const int32_t* __restrict__ parent, int B, int N,
                                                        uint64_t* __restrict__ anc, uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int32_t* par = parent + (size_t)b * N;
    int p0 = lane < N ? par[lane] : -1;
    int p1 = lane + 32 < N ? par[lane + 32] : -1;
    uint64_t m0 = 0, m1 = 0;  // this lane's nodes' masks
    bool bad = false;
    for (int i = 0; i < N; ++i) {
        const int pi = __shfl_sync(0xffffffffu, i < 32 ? p0 : p1, i & 31);
        uint64_t pm = 0;
        if (pi >= 0 && pi < i) {
            const uint64_t a0 = __shfl_sync(0xffffffffu, m0, pi & 31);
            const uint64_t a1 = __shfl_sync(0xffffffffu, m1, pi & 31);
            pm = pi < 32 ? a0 : a1;
        } else if (pi != -1) {
            bad = true;
        }
        const uint64_t mi = pm | (1ull << i);
        if ((i & 31) == lane) {
            if (i < 32) m0 = mi;
            else m1 = mi;
        }
    }
    uint64_t* out = anc + (size_t)b * N;
    if (lane < N) out[lane] = m0;
    if (lane + 32 < N) out[lane + 32] = m1;
    if (bad && lane == 0) atomicOr(status, LUCETREE_DEV_BAD_PARENT);
}

// One warp per sequence.  Lanes load the tree (node i in lane i % 32) and
// decide whether each node's draft token equals its parent row's argmax; the
// ok-flags (node and all ancestors match) and depths then follow in node
// order.  The deepest ok node (lowest id among equals: ids are scanned upward
// with a strict comparison) ends the accepted path.
__global__ void __launch_bounds__(128) accept_kernel(const int32_t* __restrict__ parent,
                                                     const int32_t* __restrict__ draft,
                                                     const int32_t* __restrict__ argmax, int B, int N, int vocab,
                                                     int32_t* __restrict__ acc_nodes, int32_t* __restrict__ acc_len,
                                                     int32_t* __restrict__ bonus, uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (b >= B) return;
    const int32_t* par = parent + (size_t)b * N;
    const int32_t* dr = draft + (size_t)b * N;
    const int32_t* am = argmax + (size_t)b * (N + 1);
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
                else match[k] = t == am[p[k] + 1];
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
    int32_t* out = acc_nodes + (size_t)b * N;
    for (int k = best_depth + lane; k < N; k += 32) out[k] = -1;
    if (lane == 0) {
        int k = best_depth;
        for (int c = best; c >= 0; c = par[c]) out[--k] = c;
        acc_len[b] = best_depth;
        bonus[b] = am[best + 1];
    }
}

// One block per sequence: 16-byte vector copies of every accepted node's K and
// V rows (all KV heads); the length update happens after the block has read
// ctx_len_in, so ctx_len_out may alias it.
__global__ void __launch_bounds__(256) commit_kernel(lucetree_commit_args c, int elem_bytes) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int L = c.ctx_len_in[b];
    const int a = c.acc_len[b];
    __shared__ int s_good;
    if (threadIdx.x == 0) s_good = 0x7fffffff;
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
        const int node = c.acc_nodes[(size_t)b * c.N + k];
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
            atomicMin(&s_good, k);
        }
    }
    __syncthreads();
    count = min(count, s_good);
    const int units = count * c.Hkv * vec_per_row;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        const int v = u % vec_per_row;
        const int g = (u / vec_per_row) % c.Hkv;
        const int k = u / (vec_per_row * c.Hkv);
        const int node = c.acc_nodes[(size_t)b * c.N + k];
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

}  // namespace

cudaError_t launch_build_anc(const int32_t* parent, int B, int N, uint64_t* anc, uint32_t* status,
                             cudaStream_t stream) {
    return launch_pdl(build_anc_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, parent, B, N, anc, status);
}

cudaError_t launch_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int B, int N,
                          int vocab, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, uint32_t* status,
                          cudaStream_t stream) {
    return launch_pdl(accept_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, parent, draft, argmax, B, N, vocab,
                      acc_nodes, acc_len, bonus, status);
}

cudaError_t launch_commit(const lucetree_commit_args& c, cudaStream_t stream) {
    return launch_pdl(commit_kernel, dim3(c.B), dim3(256), 0, stream, c, 2);
}

}  // namespace lucetree
