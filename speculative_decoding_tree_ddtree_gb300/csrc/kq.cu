// kq.cu -- tree-verify attention over K held as FP8 E4M3 codes, and the
// commit that stores accepted K rows in that format.
//
// Format (the library's own reading of the K/V quantisation the pages list
// without a layout): each (page, KV head, token) row of K is stored as D
// E4M3 codes plus one exponent byte e; the value is e4m3(code) * 2^(e - 127)
// and e = 0 reads as zero.  Storing a 16-bit row k picks the largest integer
// p with max|k| * 2^p <= 448 (E4M3's largest finite value), writes
// e = 127 - p and rounds each k * 2^p to the nearest E4M3 value, ties to the
// even code.
//
// QK runs on the FP8 tensor cores.  The prefix kernel loads each piece's
// bf16 queries (one row group of one key segment) and splits them in shared
// memory: scaled by one power of two 2^p so that their largest magnitude lies
// in (224, 448], then two E4M3 parts, hi = e4m3(q 2^p) and
// lo = e4m3(q 2^p - hi).  A bf16 query has 8 significant bits and hi keeps
// the top 4, so the residual fits lo exactly wherever it stays in E4M3's
// normal range (|q 2^p| >= 1/4); two FP8 MMAs (hi, then lo, into one fp32
// accumulator) cost one bf16 MMA.  The softmax multiplies each key's
// accumulated score by 2^(e - 127) and by scale * log2(e) / 2^p.
#include "attn_prefix_tc.cuh"
#include "e4m3.cuh"
#include "tree_ops.cuh"

namespace lucetree {

namespace {

using e4m3::e4m3x2;
using e4m3::e4m3x2_to_f32;
using e4m3::scale_exponent;

// One CTA per sequence: every accepted node's K rows (all KV heads) stored as
// E4M3 codes and exponent at logical position L_b + k, its V rows copied as
// 16-bit; ctx_len_out = L_b + count.  The entries are validated first so the
// copy stops at the first bad one (as lucetree_commit).
__global__ void __launch_bounds__(256) commit_kq_kernel(lucetree_commit_args c, uint8_t* __restrict__ k_exp) {
    __shared__ int s_good;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int L = c.ctx_len_in[b];
    const int a = c.acc_len[b];
    if (threadIdx.x == 0) s_good = 0x7fffffff;
    __syncthreads();
    int count = a;
    if (a < 0 || a > c.N || L < 0) {
        if (threadIdx.x == 0) atomicOr(c.status, a < 0 || a > c.N ? LUCETREE_DEV_BAD_NODE : LUCETREE_DEV_BAD_CTX);
        count = 0;
    }
    for (int k = threadIdx.x; k < count; k += blockDim.x) {
        const int node = c.acc_nodes[(size_t)b * c.N + k];
        const long long pos = (long long)L + k;
        const long long pi = pos / kPage;
        bool good = node >= 0 && node < c.N && pi < c.max_pages_per_seq;
        const uint32_t flag = (node >= 0 && node < c.N) ? LUCETREE_DEV_BAD_PAGE : LUCETREE_DEV_BAD_NODE;
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
    const int D = c.D;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // K: one warp per (accepted node, KV head) row, 8 dims per lane (D = 256)
    for (int r = warp; r < count * c.Hkv; r += blockDim.x / 32) {
        const int k = r / c.Hkv, g = r % c.Hkv;
        const int node = c.acc_nodes[(size_t)b * c.N + k];
        const long long pos = (long long)L + k;
        const int page = c.page_table[(size_t)b * c.max_pages_per_seq + pos / kPage];
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(c.k_tree) +
                                   (((size_t)b * c.N + node) * c.Hkv + g) * D + lane * 8;
        float v[8];
        load8_f32<__nv_bfloat16>(src, v);
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const int p = scale_exponent(m);
        const int ebyte = m > 0.f ? 127 - p : 0;
        const bool in_range = ebyte >= 1 && ebyte <= 254;  // rows outside the byte's range are stored as zero
        uint32_t w[2] = {0, 0};
        if (in_range) {
#pragma unroll
            for (int e = 0; e < 8; e += 2)
                w[e / 4] |= (uint32_t)e4m3x2(ldexpf(v[e], p), ldexpf(v[e + 1], p)) << (16 * ((e / 2) & 1));
        }
        const size_t row = ((size_t)page * c.Hkv + g) * kPage + (size_t)(pos % kPage);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(c.k_pool) + row * D + lane * 8) = make_uint2(w[0], w[1]);
        if (lane == 0) k_exp[row] = (uint8_t)(in_range ? ebyte : 0);
    }
    // V: 16-byte copies of the 16-bit rows
    const int vec_per_row = D * 2 / 16;
    const char* vt = reinterpret_cast<const char*>(c.v_tree);
    char* vp = reinterpret_cast<char*>(c.v_pool);
    const int units = count * c.Hkv * vec_per_row;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
        const int v = u % vec_per_row;
        const int g = (u / vec_per_row) % c.Hkv;
        const int k = u / (vec_per_row * c.Hkv);
        const int node = c.acc_nodes[(size_t)b * c.N + k];
        const long long pos = (long long)L + k;
        const int page = c.page_table[(size_t)b * c.max_pages_per_seq + pos / kPage];
        const size_t dst = ((((size_t)page * c.Hkv + g) * kPage + (size_t)(pos % kPage)) * D * 2) + (size_t)v * 16;
        const size_t src = ((((size_t)b * c.N + node) * c.Hkv + g) * D * 2) + (size_t)v * 16;
        *reinterpret_cast<uint4*>(vp + dst) = *reinterpret_cast<const uint4*>(vt + src);
    }
    __syncthreads();
    if (threadIdx.x == 0) c.ctx_len_out[b] = L < 0 ? L : L + count;
}

}  // namespace

lucetree_status verify_attn_check(const lucetree_attn_args* a, bool need_mask, int v_format, AttnLaunch* L);

}  // namespace lucetree

using namespace lucetree;

extern "C" lucetree_status lucetree_verify_attn_kq_workspace(int B, int N, int Hq, int Hkv, int D, size_t* bytes) {
    if (!bytes) return LUCETREE_ERR_INVALID_ARG;
    size_t attn = 0;
    const lucetree_status st = lucetree_verify_attn_workspace(B, N, Hq, Hkv, D, &attn);
    if (st != LUCETREE_OK) return st;
    if (D != 256) return LUCETREE_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LUCETREE_ERR_CUDA;
    *bytes = attn_workspace_bytes(make_plan(B, N, Hq, Hkv, D, prefix_grid_ctas(dev), 1));
    return LUCETREE_OK;
}

extern "C" lucetree_status lucetree_verify_attn_kq(const lucetree_attn_args* a, const uint8_t* k_exp, int v_format,
                                                   const uint8_t* v_exp, void* workspace, size_t workspace_bytes,
                                                   void* stream) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    if (a->dtype != LUCETREE_BF16 || a->D != 256) return LUCETREE_ERR_UNSUPPORTED;
    if (v_format != LUCETREE_V_SAME && v_format != LUCETREE_V_INT8 && v_format != LUCETREE_V_INT4)
        return LUCETREE_ERR_UNSUPPORTED;
    const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!k_exp || !al16(k_exp)) return LUCETREE_ERR_INVALID_ARG;
    if (v_format != LUCETREE_V_SAME && (!v_exp || !al16(v_exp))) return LUCETREE_ERR_INVALID_ARG;
    AttnLaunch L;
    lucetree_status st = verify_attn_check(a, true, v_format, &L);
    if (st != LUCETREE_OK) return st;
    if (!workspace || workspace_bytes < attn_workspace_bytes(L.plan) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LUCETREE_ERR_WORKSPACE;
    L.ws = reinterpret_cast<float*>(workspace);
    L.v_exp = v_format != LUCETREE_V_SAME ? v_exp : nullptr;
    L.k_format = LUCETREE_K_E4M3;
    L.k_exp = k_exp;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_attn_prefix(L, s) != cudaSuccess) return LUCETREE_ERR_CUDA;
    if (launch_attn_merge(L, s) != cudaSuccess) return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

extern "C" lucetree_status lucetree_commit_kq(const lucetree_commit_args* c, uint8_t* k_exp, void* stream) {
    if (!c || !k_exp) return LUCETREE_ERR_INVALID_ARG;
    if (c->dtype != LUCETREE_BF16 || c->D != 256) return LUCETREE_ERR_UNSUPPORTED;
    if (c->page_size != LUCETREE_PAGE_SIZE) return LUCETREE_ERR_UNSUPPORTED;
    if (c->B <= 0 || c->N <= 0 || c->Hkv <= 0 || c->num_pages <= 0 || c->max_pages_per_seq <= 0)
        return LUCETREE_ERR_INVALID_ARG;
    if (c->N > LUCETREE_MAX_NODES) return LUCETREE_ERR_UNSUPPORTED;
    if (!c->k_tree || !c->v_tree || !c->acc_nodes || !c->acc_len || !c->page_table || !c->ctx_len_in ||
        !c->ctx_len_out || !c->k_pool || !c->v_pool || !c->status)
        return LUCETREE_ERR_INVALID_ARG;
    const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al16(c->k_tree) || !al16(c->v_tree) || !al16(c->k_pool) || !al16(c->v_pool)) return LUCETREE_ERR_INVALID_ARG;
    if (launch_pdl(commit_kq_kernel, dim3(c->B), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), *c, k_exp) !=
        cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}
