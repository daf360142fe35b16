// argmax.cu -- per-row argmax over the vocabulary with lowest-index ties.
//
// Each row is cut into `chunks` slices handled by separate CTAs so the grid
// covers the GPU even for a couple of dozen rows.  A value and its index are
// packed into one 64-bit key: the high word is the float's bits mapped to an
// unsigned order (with -0.0 first turned into +0.0, so the two zeros tie), the
// low word is ~index; the maximum key is the maximum value at the lowest
// index.  The last CTA of a row (atomic ticket, no waiting) reduces the
// row's chunk keys and writes the index.
#include "internal.cuh"

namespace lucetree {

namespace {

constexpr int kThreads = 256;

__device__ inline unsigned long long pack_key(float x, unsigned idx) {
    if (x == 0.f) x = 0.f;  // -0.0 -> +0.0
    unsigned u = __float_as_uint(x);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(~idx);
}

__device__ inline unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

__device__ inline unsigned long long block_max(unsigned long long k, unsigned long long* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) k = umax64(k, __shfl_xor_sync(0xffffffffu, k, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = k;
    __syncthreads();
    if (warp == 0) {
        k = lane < kThreads / 32 ? red[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) k = umax64(k, __shfl_xor_sync(0xffffffffu, k, o));
    }
    return k;  // valid in thread 0
}

__global__ void __launch_bounds__(kThreads) argmax_kernel(const float* __restrict__ logits, int vocab,
                                                          long long row_stride, int chunks,
                                                          int32_t* __restrict__ out_idx,
                                                          unsigned long long* __restrict__ part,
                                                          unsigned* __restrict__ tickets) {
    __shared__ unsigned long long red[kThreads / 32];
    __shared__ bool is_last;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.y, ch = blockIdx.x;
    const long long per = (((long long)vocab + chunks - 1) / chunks + 3) / 4 * 4;  // multiple of 4 elements
    const long long k0 = ch * per;
    const long long k1 = min((long long)vocab, k0 + per);
    const float* x = logits + row * row_stride;
    unsigned long long best = 0ull;
    long long k = k0;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
        // 16-byte loads, kU in flight per thread (a chunk is about one round of them)
        constexpr int kU = 8;
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const long long q0 = k0 / 4, q1 = k1 / 4;  // full float4 groups in [k0, k1)
        long long q = q0 + threadIdx.x;
        for (; q + (kU - 1) * kThreads < q1; q += kU * kThreads) {
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) v[u] = __ldg(x4 + q + u * kThreads);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const unsigned base = (unsigned)(4 * (q + u * kThreads));
                best = umax64(best, pack_key(v[u].x, base));
                best = umax64(best, pack_key(v[u].y, base + 1));
                best = umax64(best, pack_key(v[u].z, base + 2));
                best = umax64(best, pack_key(v[u].w, base + 3));
            }
        }
        for (; q < q1; q += kThreads) {
            const float4 v = __ldg(x4 + q);
            const unsigned base = (unsigned)(4 * q);
            best = umax64(best, pack_key(v.x, base));
            best = umax64(best, pack_key(v.y, base + 1));
            best = umax64(best, pack_key(v.z, base + 2));
            best = umax64(best, pack_key(v.w, base + 3));
        }
        k = q1 * 4 + threadIdx.x;  // ragged tail (vocab not a multiple of 4)
    } else {
        k = k0 + threadIdx.x;
    }
    for (; k < k1; k += kThreads) best = umax64(best, pack_key(__ldg(x + k), (unsigned)k));
    best = block_max(best, red);
    if (threadIdx.x == 0) {
        part[(size_t)row * chunks + ch] = best;
        __threadfence();
        const unsigned t = atomicAdd(&tickets[row], 1u);
        is_last = (t == (unsigned)chunks - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    unsigned long long m = 0ull;
    for (int c = threadIdx.x; c < chunks; c += kThreads) m = umax64(m, __ldcg(part + (size_t)row * chunks + c));
    __syncthreads();
    m = block_max(m, red);
    if (threadIdx.x == 0) {
        out_idx[row] = (int32_t)(~(unsigned)(m & 0xffffffffull));
        tickets[row] = 0u;
    }
}

int argmax_chunks(int rows, int vocab, int device) {
    const int sms = device_sm_count(device);
    int chunks = (4 * sms + rows - 1) / rows;
    const int max_by_size = (vocab + 4 * kThreads - 1) / (4 * kThreads);
    if (chunks > max_by_size) chunks = max_by_size;
    if (chunks < 1) chunks = 1;
    return chunks;
}

}  // namespace

size_t argmax_workspace_bytes(int rows, int vocab, int device) {
    const int chunks = argmax_chunks(rows, vocab, device);
    size_t t = ((size_t)rows * sizeof(unsigned) + 255) / 256 * 256;
    return t + (size_t)rows * chunks * sizeof(unsigned long long);
}

cudaError_t launch_argmax(const float* logits, int rows, int vocab, long long row_stride, int32_t* out_idx,
                          void* ws, int device, cudaStream_t stream) {
    const int chunks = argmax_chunks(rows, vocab, device);
    unsigned* tickets = reinterpret_cast<unsigned*>(ws);
    size_t t = ((size_t)rows * sizeof(unsigned) + 255) / 256 * 256;
    unsigned long long* part = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + t);
    cudaError_t e = cudaMemsetAsync(tickets, 0, (size_t)rows * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    dim3 grid(chunks, rows);
    return launch_pdl(argmax_kernel, grid, dim3(kThreads), 0, stream, logits, vocab, row_stride, chunks, out_idx,
                      part, tickets);
}

}  // namespace lucetree
