// argmax.cuh -- per-row argmax over the vocabulary with lowest-index ties, as
// a CTA-wide device routine shared by the argmax kernel and the fused step.
//
// Each row is cut into `chunks` slices handled by separate CTAs so the grid
// covers the GPU even for a couple of dozen rows.  A value and its index are
// packed into one 64-bit key: the high word is the float's bits mapped to an
// unsigned order (with -0.0 first turned into +0.0, so the two zeros tie), the
// low word is ~index; the maximum key is the maximum value at the lowest
// index.  The last CTA of a row (atomic ticket, no waiting) reduces the
// row's chunk keys, writes the index and resets the ticket.
#pragma once

#include "internal.cuh"

namespace lucetree {
namespace am {

constexpr int kThreads = 256;
constexpr int kU = 8;  // 16-byte loads in flight per thread

__device__ inline unsigned long long pack_key(float x, unsigned idx) {
    if (x == 0.f) x = 0.f;  // -0.0 -> +0.0
    unsigned u = __float_as_uint(x);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(~idx);
}

__device__ inline unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

// Maximum over the CTA (kThreads threads); valid in thread 0.
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
    return k;
}

// Elements per chunk: a multiple of 4, so every chunk but the last starts on
// a 16-byte boundary of an aligned row.
__host__ __device__ inline long long chunk_elems(int vocab, int chunks) {
    return (((long long)vocab + chunks - 1) / chunks + 3) / 4 * 4;
}

// Chunk `ch` of row `row`, by the whole CTA.  The CTA that completes the row
// writes out_idx[row]; the return value (the same in every thread) says
// whether this CTA was that one.  s_red: kThreads / 32 keys of shared memory;
// s_flag: one shared int.
__device__ inline bool argmax_chunk(const float* __restrict__ logits, int vocab, long long row_stride, int chunks,
                                    int row, int ch, int32_t* __restrict__ out_idx,
                                    unsigned long long* __restrict__ part, unsigned* __restrict__ tickets,
                                    unsigned long long* s_red, int* s_flag) {
    const long long per = chunk_elems(vocab, chunks);
    const long long k0 = ch * per;
    const long long k1 = min((long long)vocab, k0 + per);
    const float* x = logits + row * row_stride;
    unsigned long long best = 0ull;
    long long k = k0;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
        // all of a thread's 16-byte loads of one round are issued before any is used
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const long long q1 = k1 / 4;  // full float4 groups in [k0, k1)
        for (long long q = k0 / 4 + threadIdx.x; q < q1; q += (long long)kU * kThreads) {
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u)
                v[u] = q + u * kThreads < q1 ? __ldcg(x4 + q + u * kThreads)
                                             : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (q + u * kThreads >= q1) continue;
                const unsigned base = (unsigned)(4 * (q + u * kThreads));
                best = umax64(best, pack_key(v[u].x, base));
                best = umax64(best, pack_key(v[u].y, base + 1));
                best = umax64(best, pack_key(v[u].z, base + 2));
                best = umax64(best, pack_key(v[u].w, base + 3));
            }
        }
        k = q1 * 4 > k0 ? q1 * 4 + threadIdx.x : k0 + threadIdx.x;  // ragged tail (vocab not a multiple of 4)
    } else {
        k = k0 + threadIdx.x;
    }
    for (; k < k1; k += kThreads) best = umax64(best, pack_key(__ldcg(x + k), (unsigned)k));
    best = block_max(best, s_red);
    if (threadIdx.x == 0) {
        part[(size_t)row * chunks + ch] = best;
        __threadfence();
        const unsigned t = atomicAdd(&tickets[row], 1u);
        *s_flag = (t == (unsigned)chunks - 1u);
    }
    __syncthreads();
    const bool last = *s_flag != 0;
    if (!last) return false;
    __threadfence();
    unsigned long long m = 0ull;
    for (int c = threadIdx.x; c < chunks; c += kThreads) m = umax64(m, __ldcg(part + (size_t)row * chunks + c));
    __syncthreads();  // s_red is reused
    m = block_max(m, s_red);
    if (threadIdx.x == 0) {
        out_idx[row] = (int32_t)(~(unsigned)(m & 0xffffffffull));
        tickets[row] = 0u;
    }
    return true;
}

// Chunks per row: about four CTAs per SM over all rows, and no chunk smaller
// than one round of loads.
inline int argmax_chunks(int rows, int vocab, int sms, int ctas_per_sm = 4) {
    int chunks = (ctas_per_sm * sms + rows - 1) / rows;
    const int max_by_size = (vocab + 4 * kThreads - 1) / (4 * kThreads);
    if (chunks > max_by_size) chunks = max_by_size;
    if (chunks < 1) chunks = 1;
    return chunks;
}

}  // namespace am
}  // namespace lucetree
