// verify_step.cu -- lucetree_verify_step: one whole verify step in two
// launches on the caller's stream.
//
//   1. the split-K prefix kernel of lucetree_verify_attn (tensor cores);
//   2. the "finish" kernel, a programmatic dependent of 1, with two kinds of
//      CTA in one grid:
//      - argmax CTAs (first in the grid): chunk c of logits row r.  They read
//        only the step's inputs, so they run while the prefix kernel's last
//        CTAs are still streaming K/V.  The CTA that completes a row bumps its
//        sequence's ticket; the CTA that completes the sequence's last row
//        accepts that sequence (one warp), waits for the prefix kernel to
//        complete (its reads of the pool are over) and commits the accepted
//        K/V rows with the whole CTA.
//      - merge CTAs: one per attention output row, the tree block with the
//        node's ancestors walked from the parent array, then the log-sum-exp
//        merge of the prefix partials (after waiting for the prefix kernel).
//
// The ancestor masks, the argmax, acceptance and commit therefore need no
// launches of their own.  No CTA waits on another: the tickets are atomic
// counters and only the CTA that takes the last one goes on.
#include "argmax.cuh"
#include "attn_merge.cuh"
#include "tree_ops.cuh"

namespace lucetree {

namespace {

struct StepLaunch {
    AttnLaunch attn;
    const int32_t* parent;
    const int32_t* draft;
    const float* logits;
    int vocab;
    int chunks;      // argmax chunks per logits row
    int32_t* argmax;
    int32_t* acc_nodes;
    int32_t* acc_len;
    int32_t* bonus;
    unsigned* row_tickets;           // [B * (N + 1)], zero between calls
    unsigned* seq_tickets;           // [B], zero between calls
    unsigned long long* chunk_keys;  // [B * (N + 1)][chunks]
    lucetree_commit_args commit;
};

constexpr int kThreads = 256;
// Argmax CTAs per SM's worth of logits.  They are blocks of this kernel, so
// they take a merge block's registers (two blocks per SM): the fewer they
// are, the sooner the merge blocks are resident.
constexpr int kArgmaxCtasPerSm = 2;
constexpr int kMergeWarps = 4;                         // warps per output row, as in the merge launch
constexpr int kRowsPerCta = kThreads / 32 / kMergeWarps;  // a merge CTA merges two rows side by side
static_assert(kThreads == am::kThreads, "one CTA size for every part");

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) finish_kernel(const StepLaunch S) {
    __shared__ float s_o[kRowsPerCta][kMergeWarps][D];
    __shared__ float s_red[kRowsPerCta][kMergeWarps];
    __shared__ unsigned long long s_key[kThreads / 32];
    __shared__ int32_t s_par[kRowsPerCta][LUCETREE_MAX_NODES];
    __shared__ int s_flag, s_good;
    if (threadIdx.x == 0) pdl_trigger();

    const PlanDims& p = S.attn.plan;
    const int N = p.N;
    const long long n_am = (long long)p.B * (N + 1) * S.chunks;
    if ((long long)blockIdx.x < n_am) {
        // ---------------------------------------------------------------- argmax chunk
        const int row = (int)(blockIdx.x / S.chunks), ch = (int)(blockIdx.x % S.chunks);
        if (!am::argmax_chunk(S.logits, S.vocab, S.vocab, S.chunks, row, ch, S.argmax, S.chunk_keys,
                              S.row_tickets, s_key, &s_flag))
            return;
        // this CTA completed row `row`; the sequence's last row starts acceptance
        const int b = row / (N + 1);
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned t = atomicAdd(&S.seq_tickets[b], 1u);
            s_flag = t == (unsigned)N;
            if (t == (unsigned)N) S.seq_tickets[b] = 0u;
        }
        __syncthreads();
        if (!s_flag) return;
        __threadfence();
        if (threadIdx.x < 32)
            tree::accept_warp(S.parent + (size_t)b * N, S.draft + (size_t)b * N, S.argmax + (size_t)b * (N + 1), N,
                              S.vocab, S.acc_nodes + (size_t)b * N, S.acc_len + b, S.bonus + b, S.attn.a.status);
        __syncthreads();
        // the prefix kernel reads whole pages, the rows past the committed length
        // included (they are masked): write the pool only once it has completed
        pdl_wait();
        tree::commit_block(S.commit, b, (int)sizeof(T), &s_good);
        return;
    }
    // -------------------------------------------------------------------- merge rows
    // warp group grp (kMergeWarps warps, named barrier 1 + grp) merges one row
    const int grp = (threadIdx.x >> 5) / kMergeWarps;
    const int gt = threadIdx.x - 32 * kMergeWarps * grp;
    const long long row = ((long long)blockIdx.x - n_am) * kRowsPerCta + grp;
    if (row >= (long long)p.B * N * p.Hq) return;  // (the group's barriers involve only its own warps)
    const int i = (int)((row / p.Hq) % N);
    const int b = (int)(row / ((long long)p.Hq * N));
    if (gt < N) s_par[grp][gt] = __ldcg(S.parent + (size_t)b * N + gt);
    static_assert(kRowsPerCta == 2, "two warp groups: named barriers 1 and 2");
    if (grp == 0) merge::group_sync(1, 32 * kMergeWarps);
    else merge::group_sync(2, 32 * kMergeWarps);
    bool bad = false;
    const uint64_t anc = tree::anc_walk(s_par[grp], i, &bad);
    if (bad && gt == 0 && (row % p.Hq) == 0) atomicOr(S.attn.a.status, LUCETREE_DEV_BAD_PARENT);
    if (grp == 0) merge::merge_row<T, D, kMergeWarps, 1>(S.attn, row, anc, s_o[0], s_red[0], 0);
    else merge::merge_row<T, D, kMergeWarps, 2>(S.attn, row, anc, s_o[1], s_red[1], kMergeWarps);
}

template <typename T, int D>
cudaError_t launch_finish(const StepLaunch& S, cudaStream_t stream) {
    const long long rows = (long long)S.attn.plan.B * S.attn.plan.N * S.attn.plan.Hq;
    const long long blocks = (long long)S.attn.plan.B * (S.attn.plan.N + 1) * S.chunks +
                             (rows + kRowsPerCta - 1) / kRowsPerCta;
    return launch_pdl(finish_kernel<T, D>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, S);
}

// Workspace layout after the attention partials: row tickets, sequence
// tickets (each padded to 256 bytes), then the argmax chunk keys.
struct StepWs {
    size_t attn, row_t, seq_t, keys, total;
};

StepWs step_ws(const PlanDims& p, int vocab, int sms) {
    const int rows = p.B * (p.N + 1);
    const int chunks = am::argmax_chunks(rows, vocab, sms, kArgmaxCtasPerSm);
    StepWs w;
    w.attn = (attn_workspace_bytes(p) + 255) / 256 * 256;
    w.row_t = w.attn;
    w.seq_t = w.row_t + ((size_t)rows * 4 + 255) / 256 * 256;
    w.keys = w.seq_t + ((size_t)p.B * 4 + 255) / 256 * 256;
    w.total = w.keys + (size_t)rows * chunks * 8;
    return w;
}

}  // namespace

// entry points (declared in lucetree.h)
lucetree_status verify_attn_check(const lucetree_attn_args* a, bool need_mask, int v_format, AttnLaunch* L);

}  // namespace lucetree

using namespace lucetree;

extern "C" lucetree_status lucetree_verify_step_workspace(int B, int N, int Hq, int Hkv, int D, int vocab,
                                                          size_t* bytes) {
    if (!bytes || vocab <= 0) return LUCETREE_ERR_INVALID_ARG;
    size_t attn = 0;
    const lucetree_status st = lucetree_verify_attn_workspace(B, N, Hq, Hkv, D, &attn);
    if (st != LUCETREE_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LUCETREE_ERR_CUDA;
    const PlanDims p = make_plan(B, N, Hq, Hkv, D, prefix_grid_ctas(dev), 1);
    *bytes = step_ws(p, vocab, device_sm_count(dev)).total;
    return LUCETREE_OK;
}

extern "C" lucetree_status lucetree_verify_step(const lucetree_step_args* s, void* workspace, size_t workspace_bytes,
                                                void* stream) {
    if (!s) return LUCETREE_ERR_INVALID_ARG;
    StepLaunch S;
    lucetree_status st = verify_attn_check(&s->attn, false, LUCETREE_V_SAME, &S.attn);
    if (st != LUCETREE_OK) return st;
    const lucetree_attn_args& a = s->attn;
    if (!s->parent || !s->draft || !s->logits || !s->argmax || !s->acc_nodes || !s->acc_len || !s->bonus ||
        !s->ctx_len_out || s->vocab <= 0)
        return LUCETREE_ERR_INVALID_ARG;
    if (s->ctx_len_out == a.ctx_len) return LUCETREE_ERR_INVALID_ARG;  // merge CTAs still read the old lengths
    if ((long long)a.B * (a.N + 1) > 65535) return LUCETREE_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LUCETREE_ERR_CUDA;
    const StepWs w = step_ws(S.attn.plan, s->vocab, device_sm_count(dev));
    if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return LUCETREE_ERR_WORKSPACE;
    char* ws = reinterpret_cast<char*>(workspace);
    S.attn.ws = reinterpret_cast<float*>(ws);
    S.parent = s->parent;
    S.draft = s->draft;
    S.logits = s->logits;
    S.vocab = s->vocab;
    S.chunks = am::argmax_chunks(a.B * (a.N + 1), s->vocab, device_sm_count(dev), kArgmaxCtasPerSm);
    S.argmax = s->argmax;
    S.acc_nodes = s->acc_nodes;
    S.acc_len = s->acc_len;
    S.bonus = s->bonus;
    S.row_tickets = reinterpret_cast<unsigned*>(ws + w.row_t);
    S.seq_tickets = reinterpret_cast<unsigned*>(ws + w.seq_t);
    S.chunk_keys = reinterpret_cast<unsigned long long*>(ws + w.keys);
    lucetree_commit_args& c = S.commit;
    c.dtype = a.dtype;
    c.B = a.B;
    c.N = a.N;
    c.Hkv = a.Hkv;
    c.D = a.D;
    c.page_size = a.page_size;
    c.k_tree = a.k_tree;
    c.v_tree = a.v_tree;
    c.acc_nodes = s->acc_nodes;
    c.acc_len = s->acc_len;
    c.page_table = a.page_table;
    c.max_pages_per_seq = a.max_pages_per_seq;
    c.num_pages = a.num_pages;
    c.ctx_len_in = a.ctx_len;
    c.ctx_len_out = s->ctx_len_out;
    c.k_pool = const_cast<void*>(a.k_pool);
    c.v_pool = const_cast<void*>(a.v_pool);
    c.status = a.status;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    if (launch_attn_prefix(S.attn, strm) != cudaSuccess) return LUCETREE_ERR_CUDA;
    cudaError_t e;
    if (a.dtype == LUCETREE_BF16)
        e = a.D == 256 ? launch_finish<__nv_bfloat16, 256>(S, strm) : launch_finish<__nv_bfloat16, 128>(S, strm);
    else
        e = a.D == 256 ? launch_finish<__half, 256>(S, strm) : launch_finish<__half, 128>(S, strm);
    return e == cudaSuccess ? LUCETREE_OK : LUCETREE_ERR_CUDA;
}
