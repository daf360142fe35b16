// internal.cuh -- shared definitions of the lucetree CUDA library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "lucetree.h"

namespace lucetree {

// ---------------------------------------------------------------------------
// Split plan of the committed-prefix attention.
//
// Query rows of one (sequence b, KV head g) are the N*G pairs (node i, head
// h' in the group).  They are cut into NG row groups of NPG consecutive nodes
// so a group has at most kRowsMax rows (the tensor-core tile's N extent).
// A "key segment" is one (b, g), s = b * Hkv + g, owning ceil(L_b / kTileKeys)
// key tiles.  Concatenating the segments' tiles gives a flat list of T tiles.
// The grid is NG sub-grids of Cg CTAs; CTA c of sub-grid rg takes tiles
// [floor(c*T/Cg), floor((c+1)*T/Cg)) for row group rg, so the NG CTAs that
// need the same K/V tiles stream them at the same time.  A CTA writes one
// partial (O, max, sum) per key segment its range touches, into workspace slot
// rg * (Cg + S - 1) + c + s; (c, s) is unique because both partitions are
// ordered, so Cg + S - 1 slots per row group always suffice.
// ---------------------------------------------------------------------------
constexpr int kTileKeys = 128;  // keys per tile: two 64-token pages
constexpr int kRowsMax = 144;   // rows per CTA (multiple of 16)
constexpr int kPage = LUCETREE_PAGE_SIZE;

struct RowGroups {
    int NG;   // number of row groups
    int NPG;  // nodes per group (the last group may hold fewer)
    int RG;   // rows per group = NPG * G
};

__host__ __device__ inline RowGroups make_row_groups(int N, int G) {
    RowGroups r;
    r.NG = (N * G + kRowsMax - 1) / kRowsMax;
    if (r.NG < 1) r.NG = 1;
    r.NPG = (N + r.NG - 1) / r.NG;
    while (r.NPG * G > kRowsMax && r.NPG > 1) {
        r.NG += 1;
        r.NPG = (N + r.NG - 1) / r.NG;
    }
    r.NG = (N + r.NPG - 1) / r.NPG;  // no empty trailing group
    r.RG = r.NPG * G;
    return r;
}

struct PlanDims {
    int B, N, Hq, Hkv, D, G;
    RowGroups rg;
    int S;          // key segments = B * Hkv
    int Cg;         // CTAs per row group
    int max_pages;  // page-table row length
};

__host__ __device__ inline PlanDims make_plan(int B, int N, int Hq, int Hkv, int D, int ctas, int max_pages) {
    PlanDims p;
    p.B = B; p.N = N; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.G = Hq / Hkv;
    p.rg = make_row_groups(N, p.G);
    p.S = B * Hkv;
    p.Cg = ctas / p.rg.NG;
    if (p.Cg < 1) p.Cg = 1;
    p.max_pages = max_pages;
    return p;
}

__host__ __device__ inline int grid_ctas(const PlanDims& p) { return p.Cg * p.rg.NG; }

// floats per workspace slot: O [RG][D], then max [RG], then sum [RG]; the
// stride is rounded up to 256 bytes so every slot starts 16-byte aligned
__host__ __device__ inline size_t slot_floats(const PlanDims& p) {
    return ((size_t)p.rg.RG * (p.D + 2) + 63) / 64 * 64;
}

__host__ __device__ inline size_t slot_index(const PlanDims& p, int rg, int c, int s) {
    return (size_t)rg * (p.Cg + p.S - 1) + c + s;
}

__host__ __device__ inline size_t attn_workspace_bytes(const PlanDims& p) {
    return (size_t)p.rg.NG * (p.Cg + p.S - 1) * slot_floats(p) * sizeof(float);
}

// Committed length used by the kernels: out-of-range values count as 0.
__device__ inline int seq_len(const int32_t* ctx_len, int b, int max_pages, uint32_t* status) {
    int L = ctx_len[b];
    if (L < 0 || (long long)L > (long long)max_pages * kPage) {
        if (status) atomicOr(status, LUCETREE_DEV_BAD_CTX);
        return 0;
    }
    return L;
}

__device__ inline int seq_len_quiet(const int32_t* ctx_len, int b, int max_pages) {
    int L = ctx_len[b];
    if (L < 0 || (long long)L > (long long)max_pages * kPage) return 0;
    return L;
}

__device__ inline long long tiles_of(int L) { return (L + kTileKeys - 1) / kTileKeys; }

// Total flat tiles over all key segments.
__device__ inline long long total_tiles(const PlanDims& p, const int32_t* ctx_len) {
    long long t = 0;
    for (int b = 0; b < p.B; ++b) t += tiles_of(seq_len_quiet(ctx_len, b, p.max_pages));
    return t * p.Hkv;
}

// Flat offset of key segment s's first tile.
__device__ inline long long segment_offset(const PlanDims& p, const int32_t* ctx_len, int s) {
    const int b = s / p.Hkv, g = s % p.Hkv;
    long long off = 0;
    for (int bb = 0; bb < b; ++bb) off += tiles_of(seq_len_quiet(ctx_len, bb, p.max_pages)) * p.Hkv;
    return off + (long long)g * tiles_of(seq_len_quiet(ctx_len, b, p.max_pages));
}

__device__ inline long long cta_begin(long long c, long long T, int C) { return c * T / C; }

// The CTA whose range holds flat tile t (largest c with cta_begin(c) <= t).
__device__ inline int cta_of_tile(long long t, long long T, int C) {
    return (int)(((t + 1) * (long long)C - 1) / T);
}

// ---------------------------------------------------------------------------
// 16-bit element helpers
// ---------------------------------------------------------------------------
template <typename T>
__device__ inline float to_f32(T x);
template <>
__device__ inline float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ inline float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 consecutive 16-bit elements (16 bytes) to fp32
template <typename T>
__device__ inline void load8_f32(const T* p, float* out);
template <>
__device__ inline void load8_f32<__half>(const __half* p, float* out) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 f = __half22float2(h[k]);
        out[2 * k] = f.x;
        out[2 * k + 1] = f.y;
    }
}
template <>
__device__ inline void load8_f32<__nv_bfloat16>(const __nv_bfloat16* p, float* out) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float2 f = __bfloat1622float2(h[k]);
        out[2 * k] = f.x;
        out[2 * k + 1] = f.y;
    }
}

template <typename T>
__device__ inline void load4_f32(const T* p, float* out) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = to_f32<T>(e[k]);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// launchers (each returns cudaGetLastError() of its launch)
// ---------------------------------------------------------------------------
struct AttnLaunch {
    lucetree_attn_args a;
    PlanDims plan;
    float* ws;
    float scale_log2;    // scale * log2(e)
    int v_format;        // LUCETREE_V_SAME (v_pool in dtype), LUCETREE_V_INT8 or LUCETREE_V_INT4 (v_pool holds codes)
    const uint8_t* v_exp;  // per-token exponents of quantised V [num_pages][Hkv][64]
    int k_format;          // LUCETREE_K_SAME, or LUCETREE_K_E4M3 (k_pool holds E4M3 codes)
    const uint8_t* k_exp;  // per-token exponents of E4M3 K [num_pages][Hkv][64]
};

int prefix_grid_ctas(int device);  // persistent grid size of the prefix kernel
bool prefix_shape_supported(const lucetree_attn_args& a);
cudaError_t launch_attn_prefix(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_attn_merge(const AttnLaunch& L, cudaStream_t stream);
cudaError_t launch_build_anc(const int32_t* parent, int B, int N, uint64_t* anc, uint32_t* status,
                             cudaStream_t stream);
cudaError_t launch_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int B, int N,
                          int vocab, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, uint32_t* status,
                          cudaStream_t stream);
cudaError_t launch_commit(const lucetree_commit_args& c, cudaStream_t stream);
size_t argmax_workspace_bytes(int rows, int vocab, int device);
cudaError_t launch_argmax(const float* logits, int rows, int vocab, long long row_stride, int32_t* out_idx,
                          void* ws, int device, cudaStream_t stream);

int device_sm_count(int device);

// ---------------------------------------------------------------------------
// Host helpers shared by the launchers.  Calls may come from several host
// threads, so every lazily filled cache is atomic or a thread-safe static.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 128;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, resolved from the driver once per process (null
// when the driver does not provide it).
EncodeTiledFn tensor_map_encoder();

// Per-device record of the CUDA context in which a kernel's dynamic
// shared-memory limit was last raised (0 = never).
typedef std::atomic<unsigned long long> SmemLimitSeen[kMaxDevices];

// Raises `kernel`'s dynamic shared-memory limit to `bytes` in the current
// context.  The attribute belongs to the context's copy of the module, so it
// is set again whenever the calling thread's context differs from the one
// recorded for this device (another device, or a context made after a device
// reset).  `bytes` must be the largest amount any launch of the kernel uses.
cudaError_t raise_smem_limit(const void* kernel, int bytes, SmemLimitSeen& seen);

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every library kernel is launched so that it
// may start while the previous kernel on the stream finishes; it executes
// pdl_wait() (wait until the previous grid has completed and its writes are
// visible) before its first read of global memory, and pdl_trigger() to let
// the next kernel start.  Completion stays transitive: a kernel completes only
// after its own wait returned.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace lucetree
