// argmax.cu -- lucetree_argmax: per-row argmax over the vocabulary with
// lowest-index ties (the CTA routine is in argmax.cuh).
#include "argmax.cuh"

namespace lucetree {

namespace {

__global__ void __launch_bounds__(am::kThreads) argmax_kernel(const float* __restrict__ logits, int vocab,
                                                              long long row_stride, int chunks,
                                                              int32_t* __restrict__ out_idx,
                                                              unsigned long long* __restrict__ part,
                                                              unsigned* __restrict__ tickets) {
    __shared__ unsigned long long red[am::kThreads / 32];
    __shared__ int flag;
    pdl_wait();
    pdl_trigger();
    am::argmax_chunk(logits, vocab, row_stride, chunks, blockIdx.y, blockIdx.x, out_idx, part, tickets, red, &flag);
}

}  // namespace

size_t argmax_workspace_bytes(int rows, int vocab, int device) {
    const int chunks = am::argmax_chunks(rows, vocab, device_sm_count(device));
    size_t t = ((size_t)rows * sizeof(unsigned) + 255) / 256 * 256;
    return t + (size_t)rows * chunks * sizeof(unsigned long long);
}

cudaError_t launch_argmax(const float* logits, int rows, int vocab, long long row_stride, int32_t* out_idx,
                          void* ws, int device, cudaStream_t stream) {
    const int chunks = am::argmax_chunks(rows, vocab, device_sm_count(device));
    unsigned* tickets = reinterpret_cast<unsigned*>(ws);
    size_t t = ((size_t)rows * sizeof(unsigned) + 255) / 256 * 256;
    unsigned long long* part = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(ws) + t);
    // the kernel leaves the tickets zeroed; clearing them here makes any
    // workspace usable without initialisation
    cudaError_t e = cudaMemsetAsync(tickets, 0, (size_t)rows * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
    dim3 grid(chunks, rows);
    return launch_pdl(argmax_kernel, grid, dim3(am::kThreads), 0, stream, logits, vocab, row_stride, chunks, out_idx,
                      part, tickets);
}

}  // namespace lucetree
