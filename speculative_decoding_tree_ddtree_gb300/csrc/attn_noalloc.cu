// attn_noalloc.cu -- lucetree_verify_attn_noalloc: tree-verify attention whose
// split-K scratch lives in a fixed device array owned by the library, for
// callers that cannot allocate device memory themselves.
#include <atomic>

#include "internal.cuh"

namespace lucetree {
namespace {

// Upper bound on the per-call scratch (the partial (O, max, sum) triples of the
// split-K plan).  One sequence at 24 / 4 heads, D = 256 and a 22-node tree
// needs about 21 MB on a 152-SM GPU; four sequences at 64 nodes about 27 MB.
constexpr size_t kNoAllocScratchBytes = 32u << 20;

// File-scope scratch.  Every GPU on which this library's module is loaded
// holds these 32 MiB until the process exits.  In host code the name is only
// a host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Resolves the scratch's device address on the current device (once per device).
lucetree_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LUCETREE_ERR_CUDA;
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LUCETREE_ERR_CUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return LUCETREE_OK;
}

}  // namespace
}  // namespace lucetree

extern "C" lucetree_status lucetree_verify_attn_noalloc(const lucetree_attn_args* a, void* stream) {
    if (!a) return LUCETREE_ERR_INVALID_ARG;
    size_t need = 0;
    lucetree_status st = lucetree_verify_attn_workspace(a->B, a->N, a->Hq, a->Hkv, a->D, &need);
    if (st != LUCETREE_OK) return st;
    if (need > lucetree::kNoAllocScratchBytes) return LUCETREE_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = lucetree::scratch_for_current_device(&scratch);
    if (st != LUCETREE_OK) return st;
    // The attention kernels need no zeroed scratch: every partial they read is
    // written earlier in the same call.
    return lucetree_verify_attn(a, scratch, lucetree::kNoAllocScratchBytes, stream);
}
