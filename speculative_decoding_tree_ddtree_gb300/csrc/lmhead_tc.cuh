// lmhead_tc.cuh -- lm_head projection fused with the argmax, on the tensor
// cores (tcgen05 / TMEM / TMA): the verify step needs each row's argmax of
// hidden . weight^T, not the logits, so no logit is ever written.
//
// Orientation (swap-AB, as in the attention's QK): vocabulary rows go on the
// MMA's M = 128 dimension and the R verify rows (root + tree nodes) on N,
// padded to RP (a multiple of 16):
//     D^T [128 vocab x RP] += W_chunk [128 x 64] . H_chunk^T     (K-major A and B)
// contracted over d_model in 64-wide chunks.  A CTA owns a contiguous range of
// 128-row vocabulary tiles and keeps up to 512 / RP of them in TMEM at once (a
// group); the weight streams through a ring of 16 KB chunk slots, the hidden
// states (small, reused by every group) through a ring of RP x 128 B slots.
//
// Epilogue: each of four warps reads the TMEM lanes of one quarter of a tile
// (one vocabulary row per lane, RP logits per lane), turns (logit, vocab index)
// into a 64-bit key ordered by value with the lowest index winning ties, takes
// the per-row maximum over its 32 lanes with a butterfly and folds it into a
// shared per-row maximum; after the last group the CTA folds its maxima into
// a global per-row maximum (64-bit atomicMax), and the last CTA to finish
// (atomic ticket, no waiting) writes the indices and resets the keys.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (+ TMEM owner), 2..5 = epilogue.
// Every wait is bounded; a timeout sets LUCETREE_DEV_TIMEOUT and returns.
#pragma once

#include "internal.cuh"
#include "tc_ptx.cuh"

namespace lucetree {
namespace lmhead {

using namespace tc;

constexpr int kThreads = 192;
constexpr int kVT = 128;                // vocabulary rows per tile (MMA M)
constexpr int kWChunk = kVT * 128;      // [128 vocab][64 d] 16-bit
constexpr int kSmemLimit = 227 * 1024;
constexpr int kMaxW = 16;
constexpr int kHS = 4;                  // hidden-state chunk slots
constexpr uint32_t kTmemCols = 512;

// Two CTAs per SM for up to 64 padded rows (the verify budgets): each keeps its
// own weight ring and half the tensor memory, so an SM streams two independent
// in-order rings, which keeps more of the weight in flight than one deeper ring.
// Larger row counts need the whole shared memory for their hidden-state ring.
__host__ __device__ constexpr int ctas_per_sm(int rp) { return rp <= 64 ? 2 : 1; }

struct Args {
    int rows, d_model, vocab;
    unsigned long long* keys;  // [rows] workspace, zero between calls
    unsigned* ticket;          // workspace, zero between calls
    int32_t* out_idx;
    float* out_logit;          // optional
    uint32_t* status;
};

template <int RP>
struct Layout {
    static constexpr int kCps = ctas_per_sm(RP);
    static constexpr uint32_t kTmem = kTmemCols / kCps;                         // columns this CTA owns
    static constexpr int kBudget = kCps == 1 ? kSmemLimit : 113 * 1024;        // per CTA
    static constexpr int kHBytes = RP * 128;  // one hidden-state chunk [RP rows][64 d]
    static constexpr int kTPG = (int)kTmem / RP < 16 ? (int)kTmem / RP : 16;  // tiles per TMEM fill
    static constexpr int kMiscBytes = 4096;
    static constexpr int kHOff = 0;
    static constexpr int kWOff = ((kHS * kHBytes + 1023) / 1024) * 1024;
    static constexpr int kWRaw = (kBudget - 1024 - kWOff - kMiscBytes) / kWChunk;
    static constexpr int kNW = kWRaw > kMaxW ? kMaxW : kWRaw;
    static constexpr int kMiscOff = kWOff + kNW * kWChunk;
    static constexpr int kBytes = kMiscOff + kMiscBytes + 1024;
    static_assert(kNW >= 4, "weight ring");
    static_assert(kBytes <= kBudget, "shared memory budget");
};

struct Misc {
    unsigned long long row_key[256];
    uint64_t full_w[kMaxW], empty_w[kMaxW], full_h[kHS], empty_h[kHS];
    uint64_t acc_full, acc_free, drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Misc) <= 4096, "misc region");

// (value, index) -> key: larger value first, then lower index; -0.0 == +0.0
__device__ __forceinline__ unsigned long long make_key(float x, unsigned idx) {
    if (x == 0.f) x = 0.f;
    unsigned u = __float_as_uint(x);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (unsigned long long)(~idx);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
    const unsigned u = (unsigned)(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long shfl_xor64(unsigned long long v, int m) {
    const unsigned lo = __shfl_xor_sync(0xffffffffu, (unsigned)v, m);
    const unsigned hi = __shfl_xor_sync(0xffffffffu, (unsigned)(v >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}
// Maximum of each of 16 columns over the warp's 32 lanes (recursive halving
// over lane bits 16, 8, 4, 2, then one exchange over bit 1): lanes 2c and 2c+1
// return column c's maximum.
__device__ __forceinline__ unsigned long long col_max16_u64(unsigned long long (&v)[16], int lane) {
#pragma unroll
    for (int m = 16, n = 8; m >= 2; m >>= 1, n >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const unsigned long long send = upper ? v[i] : v[i + n];
            const unsigned long long keep = upper ? v[i + n] : v[i];
            v[i] = umax64(keep, shfl_xor64(send, m));
        }
    }
    return umax64(v[0], shfl_xor64(v[0], 1));
}

__device__ __forceinline__ void set_abort(Misc* ms, uint32_t* status) {
    if (atomicExch(&ms->abort_flag, 1) == 0) atomicOr(status, LUCETREE_DEV_TIMEOUT);
}
__device__ __forceinline__ bool aborted(Misc* ms) { return *(volatile int*)&ms->abort_flag != 0; }

template <bool BF16, int RP>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(RP))
    lmhead_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_h, const Args a) {
    using Lay = Layout<RP>;
    constexpr int kTPG = Lay::kTPG;
    constexpr int kNW = Lay::kNW;
    constexpr uint32_t kAB = BF16 ? 1u : 0u;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sH = smem + Lay::kHOff;
    uint8_t* sW = smem + Lay::kWOff;
    Misc* ms = reinterpret_cast<Misc*>(smem + Lay::kMiscOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();

    const int nVT = (a.vocab + kVT - 1) / kVT;
    const int C = gridDim.x;
    const int v0 = (int)((long long)blockIdx.x * nVT / C), v1 = (int)((long long)(blockIdx.x + 1) * nVT / C);
    const int nK = a.d_model / 64;

    // ---------------------------------------------------------------- set-up
    for (int r = threadIdx.x; r < 256; r += kThreads) ms->row_key[r] = 0ull;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNW; ++i) {
            mbar_init(&ms->full_w[i], 1);
            mbar_init(&ms->empty_w[i], 1);
        }
        for (int i = 0; i < kHS; ++i) {
            mbar_init(&ms->full_h[i], 1);
            mbar_init(&ms->empty_h[i], 1);
        }
        mbar_init(&ms->acc_full, 1);
        mbar_init(&ms->acc_free, 4);
        mbar_init(&ms->drain, 1);
        ms->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&ms->tmem_base, Lay::kTmem);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_h);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            uint32_t wc = 0, hc = 0;
            bool ok = true;
            for (int g0 = v0; g0 < v1 && ok; g0 += kTPG) {
                const int nt = min(kTPG, v1 - g0);
                for (int kc = 0; kc < nK && ok; ++kc) {
                    const int hs = hc % kHS;
                    if (!(ok = mbar_wait(&ms->empty_h[hs], ((hc / kHS) & 1) ^ 1))) break;
                    mbar_arrive_expect_tx(&ms->full_h[hs], Lay::kHBytes);
                    tma_load_2d(sH + hs * Lay::kHBytes, &tm_h, 64 * kc, 0, &ms->full_h[hs]);
                    ++hc;
                    for (int t = 0; t < nt; ++t) {
                        const int ws = wc % kNW;
                        if (!(ok = mbar_wait(&ms->empty_w[ws], ((wc / kNW) & 1) ^ 1))) break;
                        mbar_arrive_expect_tx(&ms->full_w[ws], kWChunk);
                        tma_load_2d(sW + ws * kWChunk, &tm_w, 64 * kc, (g0 + t) * kVT, &ms->full_w[ws]);
                        ++wc;
                    }
                }
            }
            if (!ok || aborted(ms)) {
                set_abort(ms, a.status);
                // wait (bounded) for this CTA's own copies still in flight
                const uint32_t fw = wc > (uint32_t)kNW ? wc - kNW : 0u;
                for (uint32_t c = fw; c < wc; ++c) mbar_wait(&ms->full_w[c % kNW], (c / kNW) & 1, 200000000ll);
                const uint32_t fh = hc > (uint32_t)kHS ? hc - kHS : 0u;
                for (uint32_t c = fh; c < hc; ++c) mbar_wait(&ms->full_h[c % kHS], (c / kHS) & 1, 200000000ll);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, RP, kAB, 0, 0);
            constexpr uint64_t hi_k = desc_hi(16, 1024, kLayoutSwizzle128);
            const uint32_t aW = smem_u32(sW), aH = smem_u32(sH);
            uint32_t wc = 0, hc = 0;
            int grp = 0;
            bool ok = true;
            for (int g0 = v0; g0 < v1 && ok; g0 += kTPG, ++grp) {
                const int nt = min(kTPG, v1 - g0);
                // the epilogue has read the previous group's accumulators
                if (grp > 0 && !(ok = mbar_wait(&ms->acc_free, (grp - 1) & 1))) break;
                tc_fence_after();
                for (int kc = 0; kc < nK && ok; ++kc) {
                    const int hs = hc % kHS;
                    if (!(ok = mbar_wait(&ms->full_h[hs], (hc / kHS) & 1))) break;
                    tc_fence_after();
                    for (int t = 0; t < nt; ++t) {
                        const int ws = wc % kNW;
                        if (!(ok = mbar_wait(&ms->full_w[ws], (wc / kNW) & 1))) break;
                        tc_fence_after();
#pragma unroll
                        for (int sub = 0; sub < 4; ++sub) {
                            const uint64_t ad = make_desc(hi_k, aW + ws * kWChunk + sub * 32);
                            const uint64_t bd = make_desc(hi_k, aH + hs * Lay::kHBytes + sub * 32);
                            mma_f16_ss(tmem + t * RP, ad, bd, idesc, (kc | sub) != 0);
                        }
                        mma_commit(&ms->empty_w[ws]);
                        ++wc;
                    }
                    mma_commit(&ms->empty_h[hs]);
                    ++hc;
                }
                if (ok) mma_commit(&ms->acc_full);
            }
            if (!ok || aborted(ms)) {
                set_abort(ms, a.status);
                mma_commit(&ms->drain);  // every MMA issued so far has finished before TMEM is freed
                mbar_wait(&ms->drain, 0, 200000000ll);
            }
        }
        __syncwarp();
    } else {
        // ============================================================ epilogue
        const int quarter = warp & 3;  // warps 2..5 cover lane quarters 2, 3, 0, 1
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        bool bad = false;
        int grp = 0;
        for (int g0 = v0; g0 < v1; g0 += kTPG, ++grp) {
            const int nt = min(kTPG, v1 - g0);
            const bool w = mbar_wait(&ms->acc_full, grp & 1);
            if (!__all_sync(0xffffffffu, w)) {
                bad = true;
                break;
            }
            tc_fence_after();
            for (int t = 0; t < nt; ++t) {
                const unsigned v = (unsigned)((g0 + t) * kVT + quarter * 32 + lane);
                const bool vok = v < (unsigned)a.vocab;
#pragma unroll 1
                for (int cb = 0; cb < RP / 16; ++cb) {
                    uint32_t r[16];
                    tmem_ld16(tl + t * RP + 16 * cb, r);
                    tmem_wait_ld_regs16(r);
                    unsigned long long k[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        k[c] = (vok && 16 * cb + c < a.rows) ? make_key(__uint_as_float(r[c]), v) : 0ull;
                    const unsigned long long best = col_max16_u64(k, lane);
                    const int row = 16 * cb + (lane >> 1);
                    if ((lane & 1) == 0 && row < a.rows && best) atomicMax(&ms->row_key[row], best);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms->acc_free);
        }
        if (bad) set_abort(ms, a.status);
    }

    // ---------------------------------------------------------------- fold + finish
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, Lay::kTmem);
    for (int r = threadIdx.x; r < a.rows; r += kThreads)
        if (ms->row_key[r]) atomicMax(a.keys + r, ms->row_key[r]);
    __threadfence();
    __syncthreads();
    __shared__ bool is_last;
    if (threadIdx.x == 0) is_last = atomicAdd(a.ticket, 1u) == (unsigned)C - 1u;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    for (int r = threadIdx.x; r < a.rows; r += kThreads) {
        const unsigned long long k = atomicExch(a.keys + r, 0ull);  // read and reset for the next call
        a.out_idx[r] = k ? (int32_t)(~(unsigned)(k & 0xffffffffull)) : -1;
        if (a.out_logit) a.out_logit[r] = k ? key_value(k) : -INFINITY;
    }
    if (threadIdx.x == 0) *a.ticket = 0u;
}

}  // namespace lmhead

cudaError_t launch_lmhead_bf16(int rp, const CUtensorMap& tw, const CUtensorMap& th, const lmhead::Args& a, int ctas,
                               cudaStream_t stream);
cudaError_t launch_lmhead_f16(int rp, const CUtensorMap& tw, const CUtensorMap& th, const lmhead::Args& a, int ctas,
                              cudaStream_t stream);

}  // namespace lucetree
