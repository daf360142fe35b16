// lucetree_abi.cu -- the extern "C" entry points: argument checks, workspace
// sizing and kernel launches on the caller's stream.
#include <atomic>
#include <cstring>

#include "internal.cuh"
#include "lmhead.h"
#include "delta.h"
#include "stage.h"

namespace lucetree {

int device_sm_count(int device) {
    // calls may come from several host threads: the per-device cache is atomic
    // (two threads that both miss store the same value)
    static std::atomic<int> cache[128];
    if (device < 0 || device >= 128) return 1;
    int n = cache[device].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0) n = 1;
        cache[device].store(n, std::memory_order_relaxed);
    }
    return n;
}

EncodeTiledFn tensor_map_encoder() {
    // a function-local static is initialised exactly once even when several threads arrive together
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Process-unique id of the calling thread's current context, 0 if unknown.
unsigned long long current_context_id() {
    struct Fns {
        CtxGetCurrentFn get_current = nullptr;
        CtxGetIdFn get_id = nullptr;
    };
    static const Fns fns = []() {
        Fns f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
        return f;
    }();
    if (!fns.get_current || !fns.get_id) return 0;
    CUcontext ctx = nullptr;
    if (fns.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

cudaError_t raise_smem_limit(const void* kernel, int bytes, SmemLimitSeen& seen) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // the first runtime call may be the one that makes the primary context current
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && dev >= 0 && dev < kMaxDevices && seen[dev].load(std::memory_order_acquire) == ctx)
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    const unsigned long long now = current_context_id();
    if (now != 0 && dev >= 0 && dev < kMaxDevices) seen[dev].store(now, std::memory_order_release);
    return cudaSuccess;
}

static int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return 0;
    return d;
}

static bool attn_shape_ok(int B, int N, int Hq, int Hkv, int D) {
    if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0) return false;
    if (N > LUCETREE_MAX_NODES) return false;
    if (Hq % Hkv != 0) return false;
    if (D != 128 && D != 256) return false;
    if (Hq / Hkv > kRowsMax) return false;
    return true;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace lucetree

using namespace lucetree;

extern "C" {

int lucetree_abi_version(void) { return 1; }

const char* lucetree_status_string(lucetree_status s) {
    switch (s) {
        case LUCETREE_OK: return "ok";
        case LUCETREE_ERR_INVALID_ARG: return "invalid argument";
        case LUCETREE_ERR_UNSUPPORTED: return "unsupported shape";
        case LUCETREE_ERR_WORKSPACE: return "workspace missing or too small";
        case LUCETREE_ERR_CUDA: return "CUDA error";
        case LUCETREE_ERR_DEVICE_CHECK: return "device check failed";
        case LUCETREE_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

lucetree_status lucetree_verify_attn_workspace(int B, int N, int Hq, int Hkv, int D, size_t* bytes) {
    if (!bytes) return LUCETREE_ERR_INVALID_ARG;
    if (!attn_shape_ok(B, N, Hq, Hkv, D)) return LUCETREE_ERR_UNSUPPORTED;
    PlanDims p = make_plan(B, N, Hq, Hkv, D, prefix_grid_ctas(current_device()), 1);
    *bytes = attn_workspace_bytes(p);
    return LUCETREE_OK;
}

static lucetree_status verify_attn_impl(const lucetree_attn_args* a, int v_format, const uint8_t* v_exp,
                                        void* workspace, size_t workspace_bytes, void* stream);

lucetree_status lucetree_verify_attn(const lucetree_attn_args* a, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    return verify_attn_impl(a, LUCETREE_V_SAME, nullptr, workspace, workspace_bytes, stream);
}

lucetree_status lucetree_verify_attn_vq(const lucetree_attn_args* a, int v_format, const uint8_t* v_exp,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    if (v_format != LUCETREE_V_INT8 && v_format != LUCETREE_V_INT4) return LUCETREE_ERR_UNSUPPORTED;
    if (!v_exp || !aligned16(v_exp)) return LUCETREE_ERR_INVALID_ARG;
    if (a && a->D != 256) return LUCETREE_ERR_UNSUPPORTED;
    return verify_attn_impl(a, v_format, v_exp, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace lucetree {

// Host checks of one attention call and its launch description (everything
// but the workspace).  need_mask: whether anc_mask is read (the fused step
// derives the masks from the parent array instead).
lucetree_status verify_attn_check(const lucetree_attn_args* a, bool need_mask, int v_format, AttnLaunch* L) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    if (a->dtype != LUCETREE_F16 && a->dtype != LUCETREE_BF16) return LUCETREE_ERR_UNSUPPORTED;
    if (a->page_size != LUCETREE_PAGE_SIZE) return LUCETREE_ERR_UNSUPPORTED;
    if (!attn_shape_ok(a->B, a->N, a->Hq, a->Hkv, a->D)) return LUCETREE_ERR_UNSUPPORTED;
    if (!a->q || !a->k_pool || !a->v_pool || !a->page_table || !a->ctx_len || !a->k_tree || !a->v_tree ||
        (need_mask && !a->anc_mask) || !a->out || !a->status)
        return LUCETREE_ERR_INVALID_ARG;
    if (a->num_pages <= 0 || a->max_pages_per_seq <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k_pool) || !aligned16(a->v_pool) || !aligned16(a->k_tree) ||
        !aligned16(a->v_tree) || !aligned16(a->out))
        return LUCETREE_ERR_INVALID_ARG;
    if (!isfinite(a->scale)) return LUCETREE_ERR_INVALID_ARG;
    if (!prefix_shape_supported(*a)) return LUCETREE_ERR_UNSUPPORTED;
    const int dev = current_device();
    L->a = *a;
    L->plan = make_plan(a->B, a->N, a->Hq, a->Hkv, a->D, prefix_grid_ctas(dev), a->max_pages_per_seq);
    L->ws = nullptr;
    L->scale_log2 = a->scale * kLog2e;
    L->v_format = v_format;
    L->v_exp = nullptr;
    L->k_format = LUCETREE_K_SAME;
    L->k_exp = nullptr;
    return LUCETREE_OK;
}

}  // namespace lucetree

extern "C" {

static lucetree_status verify_attn_impl(const lucetree_attn_args* a, int v_format, const uint8_t* v_exp,
                                        void* workspace, size_t workspace_bytes, void* stream) {
    AttnLaunch L;
    const lucetree_status st = verify_attn_check(a, true, v_format, &L);
    if (st != LUCETREE_OK) return st;
    if (!workspace || workspace_bytes < attn_workspace_bytes(L.plan) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LUCETREE_ERR_WORKSPACE;
    L.ws = reinterpret_cast<float*>(workspace);
    L.v_exp = v_exp;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_attn_prefix(L, s) != cudaSuccess) return LUCETREE_ERR_CUDA;
    if (launch_attn_merge(L, s) != cudaSuccess) return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_build_anc_mask(const int32_t* parent, int B, int N, uint64_t* anc, uint32_t* status,
                                        void* stream) {
    if (!parent || !anc || !status || B <= 0 || N <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (N > LUCETREE_MAX_NODES) return LUCETREE_ERR_UNSUPPORTED;
    if (launch_build_anc(parent, B, N, anc, status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_argmax_workspace(int rows, int vocab, size_t* bytes) {
    if (!bytes || rows <= 0 || vocab <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (rows > 65535) return LUCETREE_ERR_UNSUPPORTED;
    *bytes = argmax_workspace_bytes(rows, vocab, current_device());
    return LUCETREE_OK;
}

lucetree_status lucetree_argmax(const float* logits, int rows, int vocab, long long row_stride, int32_t* out_idx,
                                void* workspace, size_t workspace_bytes, void* stream) {
    if (!logits || !out_idx || rows <= 0 || vocab <= 0 || row_stride < vocab) return LUCETREE_ERR_INVALID_ARG;
    if (rows > 65535) return LUCETREE_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (!workspace || workspace_bytes < argmax_workspace_bytes(rows, vocab, dev) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LUCETREE_ERR_WORKSPACE;
    if (launch_argmax(logits, rows, vocab, row_stride, out_idx, workspace, dev,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_lmhead_argmax_workspace(int rows, size_t* bytes) {
    if (!bytes || rows <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (lmhead_padded_rows(rows) < 0) return LUCETREE_ERR_UNSUPPORTED;
    *bytes = lmhead_workspace_bytes(rows);
    return LUCETREE_OK;
}

lucetree_status lucetree_lmhead_argmax(const lucetree_lmhead_args* a, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    if (a->dtype != LUCETREE_F16 && a->dtype != LUCETREE_BF16) return LUCETREE_ERR_UNSUPPORTED;
    if (!a->hidden || !a->weight || !a->out_idx || !a->status) return LUCETREE_ERR_INVALID_ARG;
    if (a->rows <= 0 || a->d_model <= 0 || a->vocab <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (lmhead_padded_rows(a->rows) < 0 || a->d_model % 64 != 0) return LUCETREE_ERR_UNSUPPORTED;
    if (!aligned16(a->hidden) || !aligned16(a->weight)) return LUCETREE_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < lmhead_workspace_bytes(a->rows) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LUCETREE_ERR_WORKSPACE;
    if (launch_lmhead(*a, workspace, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

static lucetree_status delta_check(const lucetree_delta_args* a, bool tree) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    if (a->dtype != LUCETREE_F16 && a->dtype != LUCETREE_BF16) return LUCETREE_ERR_UNSUPPORTED;
    if (a->B < 1 || a->N < 1 || a->Hk < 1 || a->Hv < 1 || a->Hv % a->Hk != 0 || a->B > 65535 || a->Hv > 65535)
        return LUCETREE_ERR_INVALID_ARG;
    if (a->dk != 128 || a->dv < 8 || a->dv % 8 != 0 || a->N > 64) return LUCETREE_ERR_UNSUPPORTED;
    if (!a->k || !a->v || !a->alpha || !a->beta || !a->state || !a->status) return LUCETREE_ERR_INVALID_ARG;
    if (tree && (!a->q || !a->parent || !a->out)) return LUCETREE_ERR_INVALID_ARG;
    if (!tree && (!a->acc_nodes || !a->acc_len)) return LUCETREE_ERR_INVALID_ARG;
    auto al = [](const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
    if (!al(a->k, 8) || !al(a->state, 16) || (tree && !al(a->q, 8))) return LUCETREE_ERR_INVALID_ARG;
    return LUCETREE_OK;
}

lucetree_status lucetree_delta_tree(const lucetree_delta_args* a, void* stream) {
    const lucetree_status st = delta_check(a, true);
    if (st != LUCETREE_OK) return st;
    if (launch_delta_tree(*a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_delta_commit(const lucetree_delta_args* a, void* stream) {
    const lucetree_status st = delta_check(a, false);
    if (st != LUCETREE_OK) return st;
    if (launch_delta_commit(*a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_stage_pages(const lucetree_stage_args* a, void* stream) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    if (a->n < 0 || a->Hkv < 1 || a->D < 8 || a->D % 8 != 0 || a->host_pages < 0 || a->num_pages < 1)
        return LUCETREE_ERR_INVALID_ARG;
    if (a->n == 0) return LUCETREE_OK;
    if (!a->host_k || !a->host_v || !a->src || !a->dst || !a->k_pool || !a->v_pool || !a->status)
        return LUCETREE_ERR_INVALID_ARG;
    if (a->table_idx && (!a->page_table || a->table_len < 1)) return LUCETREE_ERR_INVALID_ARG;
    if (!aligned16(a->host_k) || !aligned16(a->host_v) || !aligned16(a->k_pool) || !aligned16(a->v_pool))
        return LUCETREE_ERR_INVALID_ARG;
    // the host pools must be page-locked host memory mapped for the device
    void* hk = nullptr;
    void* hv = nullptr;
    if (cudaHostGetDevicePointer(&hk, const_cast<void*>(a->host_k), 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&hv, const_cast<void*>(a->host_v), 0) != cudaSuccess) {
        cudaGetLastError();  // the failed query leaves a (non-sticky) error behind: clear it
        return LUCETREE_ERR_INVALID_ARG;
    }
    if (!aligned16(hk) || !aligned16(hv)) return LUCETREE_ERR_INVALID_ARG;
    if (launch_stage_pages(*a, hk, hv, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int B, int N,
                                int vocab, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, uint32_t* status,
                                void* stream) {
    if (!parent || !draft || !argmax || !acc_nodes || !acc_len || !bonus || !status) return LUCETREE_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || vocab <= 0) return LUCETREE_ERR_INVALID_ARG;
    if (N > LUCETREE_MAX_NODES) return LUCETREE_ERR_UNSUPPORTED;
    if (launch_accept(parent, draft, argmax, B, N, vocab, acc_nodes, acc_len, bonus, status,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

lucetree_status lucetree_commit(const lucetree_commit_args* c, void* stream) {
    if (!c) return LUCETREE_ERR_INVALID_ARG;
    if (c->dtype != LUCETREE_F16 && c->dtype != LUCETREE_BF16) return LUCETREE_ERR_UNSUPPORTED;
    if (c->page_size != LUCETREE_PAGE_SIZE) return LUCETREE_ERR_UNSUPPORTED;
    if (c->B <= 0 || c->N <= 0 || c->Hkv <= 0 || c->D <= 0 || c->num_pages <= 0 || c->max_pages_per_seq <= 0)
        return LUCETREE_ERR_INVALID_ARG;
    if (c->N > LUCETREE_MAX_NODES) return LUCETREE_ERR_UNSUPPORTED;
    if ((c->D * 2) % 16 != 0) return LUCETREE_ERR_UNSUPPORTED;
    if (!c->k_tree || !c->v_tree || !c->acc_nodes || !c->acc_len || !c->page_table || !c->ctx_len_in ||
        !c->ctx_len_out || !c->k_pool || !c->v_pool || !c->status)
        return LUCETREE_ERR_INVALID_ARG;
    if (!aligned16(c->k_tree) || !aligned16(c->v_tree) || !aligned16(c->k_pool) || !aligned16(c->v_pool))
        return LUCETREE_ERR_INVALID_ARG;
    if (launch_commit(*c, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LUCETREE_ERR_CUDA;
    return LUCETREE_OK;
}

}  // extern "C"
