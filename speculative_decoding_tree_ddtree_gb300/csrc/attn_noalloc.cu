// attn_noalloc.cu -- lucetree_verify_attn_noalloc: tree-verify attention whose
// split-K scratch lives in a fixed device array owned by the library, for
// callers that cannot allocate device memory themselves.
#include "internal.cuh"

namespace lucetree {
namespace {

// Upper bound on the per-call scratch (the partial (O, max, sum) triples of the
// split-K plan).  One sequence at 24 / 4 heads, D = 256 and a 22-node tree
// needs about 21 MB on a 152-SM GPU; four sequences at 64 nodes about 27 MB.
constexpr size_t kNoAllocScratchBytes = LUCETREE_NOALLOC_SCRATCH_BYTES;

// File-scope scratch.  Every GPU on which this library's module is loaded
// holds these bytes until the process exits.  In host code the name is only
// a host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The scratch's device address in the calling thread's current context.  It
// is looked up on every call: the address belongs to one context's copy of
// the module, and a device reset (or another context on the same device)
// gives the array a new one.  After the first call in a context this is a
// host-side table lookup; the first one may load the module.
lucetree_status scratch_for_current_context(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();  // leave no error behind for the caller's next runtime call
        return LUCETREE_ERR_CUDA;
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
    st = lucetree::scratch_for_current_context(&scratch);
    if (st != LUCETREE_OK) return st;
    // The attention kernels need no zeroed scratch: every partial they read is
    // written earlier in the same call.
    return lucetree_verify_attn(a, scratch, lucetree::kNoAllocScratchBytes, stream);
}
