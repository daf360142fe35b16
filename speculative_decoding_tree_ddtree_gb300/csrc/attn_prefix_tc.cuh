// attn_prefix_tc.cuh -- committed-prefix part of tree-verify attention on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA-fed operands).
//
// Orientation.  Per (sequence, KV head, row group) the query rows are the
// (node, head-in-group) pairs of the group's nodes (132 at budget 22 with 6
// heads per KV head, one group).  Keys, not queries, go on the MMA's M = 128
// dimension so the rows only pad to a multiple of 16 (the MMA's N):
//     S^T [128 keys x R]  = K_tile [128 x D]  . Q^T          (K-major A and B)
//     O^T [D x R]        += V_tile^T [D x 128] . P^T [128 x R] (MN-major A and B)
// Keeping all of a KV head's rows in one CTA means each K/V tile passes
// through one SM's shared memory and tensor cores once; splitting the rows
// over several CTAs would multiply that traffic, which is what bounds this
// kernel on the SM side.
//
// TMEM (512 columns): S^T at columns [0, R), then O^T for d 0..127 and d
// 128..255.  TMEM lane l holds key l of S^T and output dim l (+128) of O^T.
//
// Operand precision.  QK runs on the input type (bf16 or fp16).  PV always
// runs on fp16: P^T is written as fp16 (11 significant bits, enough for the
// 2e-3 bar; bf16 P with its 8 bits is not), and bf16 V chunks are converted
// to fp16 in shared memory once they land, which is exact for every bf16
// value of magnitude below 65536 (the fp16 range; a larger one becomes inf
// and the merge flags the row's non-finite output).  An MMA's A and B then
// always share one type.
//
// Software pipeline.  The MMA warp issues QK(t+1) as soon as the softmax has
// released S^T(t) (after its exponent vote), before PV(t); so the scores of
// the next tile are computed on the tensor cores while the softmax stores
// P^T(t), and PV(t) follows.  The softmax of tile t starts writing P^T once
// PV(t-1) has finished reading it.  K and V chunks stream through the ring
// in that consumption order: K(0) K(1) V(0) K(2) V(1) ... K(n-1) V(n-2) V(n-1).
//
// Softmax over keys runs across TMEM lanes.  Each softmax thread owns one key
// lane and keeps per-column partial sums in registers; the shift m[r] per
// query row is stale on purpose.  A tile is first exponentiated with the
// current shifts (one streaming pass: P kept in registers, sums accumulated,
// largest exponent tracked; padding columns carry a shift of +inf, so they give
// P = 0 without a column test); if any exponent exceeds 8 (log2 domain) the pass is taken
// back out exactly, the tile's column maxima are found (warp shuffles +
// shared memory) and the partial sums and already-accumulated O^T columns are
// rescaled before the tile is redone.  The first tile of every range goes
// straight to that path.  Sums are reduced across lanes once per range.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (+ TMEM owner), 2..3 = bf16 -> fp16
// conversion of 16-bit V chunks (warpgroup 0 hands most of its registers to the
// others), 4..15 = softmax, expansion of quantised V codes, and epilogue: warp w
// reads TMEM lanes 32*(w%4) .. +31 and handles one third of the row tile's
// column chunks.  K and V stream through
// a ring of 16 KB chunk slots, two TMA boxes of [64 keys][64 d] (128-byte
// swizzle) per slot; an operand (one tile's K or V) is D/64 consecutive
// chunks.  A K chunk is [128 keys][64 d] (one box per 64-token page: the
// K-major A operand of QK for one 64-dim slice); a V chunk is [64 keys][128 d]
// (one page, two adjacent 64-dim boxes: the MN-major A operand of PV for 128
// output dims and 64 keys, the second box at a fixed 8 KB offset), so every
// chunk is self-contained and the ring may have any number of slots.  Every
// wait is bounded; a timeout sets LUCETREE_DEV_TIMEOUT, drains this CTA's own
// copies and MMAs and returns.
#pragma once

#include "e4m3.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace lucetree {
namespace prefix_tc {

using namespace tc;

constexpr int kSmGroups = 3;                        // softmax warps per TMEM lane quarter
constexpr int kConvWarps = 2;                       // warps 2, 3: 16-bit V conversion
constexpr int kSmWarps = 4 * kSmGroups;             // 12 softmax warps
constexpr int kSoftmaxThreads = 32 * kSmWarps;      // 384
constexpr int kThreads = 128 + kSoftmaxThreads;     // + warpgroup 0 (producer, MMA, two idle warps)
// Register split (setmaxnreg): the block is launched with 128 per thread
// (65536 / 512); warpgroup 0 gives back down to kRegsIssue and the three
// softmax warpgroups take kRegsSoftmax.  4*32*56 + 12*32*152 = 65536.
constexpr uint32_t kRegsIssue = 56, kRegsSoftmax = 152;
static_assert(kThreads == 512, "register split assumes 16 warps");
static_assert(128 * kRegsIssue + kSoftmaxThreads * kRegsSoftmax <= 65536, "register split exceeds the launch");

constexpr int kChunkBytes = 128 * 128;
constexpr int kSmemLimit = 227 * 1024;
constexpr float kTau = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSlots = 12;
static_assert(3 * kRowsMax <= (int)kTmemCols, "S^T and two O^T halves in TMEM");

template <int D, int RGP>
struct Layout {
    static constexpr int kChunks = D / 64;
    static constexpr int kDh = D / 128;                 // O^T halves of 128 output dims
    static constexpr int kNch = RGP / 16;
    static constexpr int kQBytes = kChunks * RGP * 128;
    static constexpr int kPBytes = RGP * 256;           // P^T [128 keys][RGP] fp16
    static constexpr uint32_t kColO0 = RGP;             // O^T, d 0..127
    static constexpr uint32_t kColO1 = 2 * RGP;         // O^T, d 128..255
    static_assert(RGP + kDh * RGP <= (int)kTmemCols, "TMEM columns");
    static constexpr int kMiscBytes = 5632;
    static constexpr int kRaw = (kSmemLimit - 1024 - kQBytes - kPBytes - kMiscBytes) / kChunkBytes;
    static constexpr int kNS = kRaw > kMaxSlots ? kMaxSlots : kRaw;
    static constexpr int kQOff = 0;
    static constexpr int kPOff = kQBytes;
    static constexpr int kSlotOff = ((kPOff + kPBytes + 1023) / 1024) * 1024;
    static constexpr int kMiscOff = kSlotOff + kNS * kChunkBytes;
    // force one CTA per SM: the kernel owns all 512 TMEM columns
    static constexpr int kBytesRaw = kMiscOff + kMiscBytes + 1024;
    static constexpr int kBytes = kBytesRaw < 120 * 1024 ? 120 * 1024 : kBytesRaw;
    static_assert(kNS >= kChunks, "the K/V ring must hold one whole operand");
    static_assert(kBytes <= kSmemLimit, "shared memory budget");
};

struct Misc {
    // quantised V: the per-token exponents of V chunk n at [n % kMaxSlots]; each row is a
    // TMA destination, which must be 128-byte aligned (the misc region is 1024-aligned)
    alignas(128) uint8_t vexp[kMaxSlots][128];
    alignas(16) float m_ref[kRowsMax];
    alignas(16) float alpha[kRowsMax];
    alignas(16) float col_red[4][kRowsMax];
    uint64_t full[kMaxSlots];
    uint64_t empty[kMaxSlots];
    // V chunks have their own barriers, indexed by V chunk number n (in V
    // order) modulo kMaxSlots >= kNS: vfull[n % kMaxSlots] = landed,
    // vready[n % kMaxSlots] = made the fp16 operand (16-bit V by warps 2 and 3,
    // quantised V by the softmax warps).  full[slot] still
    // completes one phase per fill (a plain arrive for V fills), so the K
    // waits' parities keep counting fills.
    uint64_t vfull[kMaxSlots];
    uint64_t vready[kMaxSlots];
    uint64_t s_full, s_free, q_full, q_empty, p_full, pv_done, drain;
    uint64_t q_ready;  // E4M3 K: the piece's queries split into their two E4M3 parts
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Misc) <= 5632, "misc region");
static_assert(offsetof(Misc, vexp) == 0 && sizeof(Misc::vexp[0]) % 128 == 0, "128-byte aligned TMA destinations");

// Quantised V (VQ = 1: int8 codes, VQ = 2: int4 codes two per byte, low
// nibble first), value = code * 2^(e - 127) with one exponent byte e per
// token.  A V chunk's codes ([64 keys][128 dims]) land at the back of its
// 16 KB slot and are expanded to the fp16 operand over the whole slot.
template <int VQ>
struct VCodes {
    static constexpr int kRowBytes = VQ == 1 ? 128 : 64;       // one key's 128 dims
    static constexpr int kBytes = kRowBytes * kPage;             // 8 KB / 4 KB
    static constexpr int kOff = kChunkBytes - kBytes;
};

// A key segment's share of this CTA's tiles.  Tile indices are 32-bit: the
// host refuses shapes whose flat tile count reaches 2^31.
struct Piece {
    int s, L;    // key segment (b * Hkv + g) and its committed length
    int ta, te;  // tile range within the segment
};

struct PieceIter {
    int t0, t1, off, s;
    __device__ bool next(const PlanDims& p, const int32_t* ctx_len, Piece& out) {
        while (s < p.S && off < t1) {
            const int L = seq_len_quiet(ctx_len, s / p.Hkv, p.max_pages);
            const int s0 = off, s1 = off + (int)tiles_of(L);
            const int cur = s;
            off = s1;
            ++s;
            if (s1 == s0 || s1 <= t0) continue;
            out.s = cur;
            out.L = L;
            out.ta = (t0 > s0 ? t0 : s0) - s0;
            out.te = (t1 < s1 ? t1 : s1) - s0;
            return true;
        }
        return false;
    }
};

// The CTA's tiles in order: piece (key segment) and tile within the segment.
struct TileCursor {
    PieceIter it;
    Piece pc;
    int t;
    int piece_no;
    bool live;
    __device__ void start(int t0, int t1, const PlanDims& p, const int32_t* ctx_len) {
        it = PieceIter{t0, t1, 0, 0};
        piece_no = -1;
        t = 0;
        next_piece(p, ctx_len);
    }
    __device__ void next_piece(const PlanDims& p, const int32_t* ctx_len) {
        live = it.next(p, ctx_len, pc);
        if (live) {
            t = pc.ta;
            ++piece_no;
        }
    }
    __device__ bool first() const { return t == pc.ta; }
    __device__ bool last() const { return t == pc.te - 1; }
    __device__ void step(const PlanDims& p, const int32_t* ctx_len) {
        if (++t >= pc.te) next_piece(p, ctx_len);
    }
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Column maxima of a warp's 16 x 32 values (v[k] = column k in this lane):
// recursive halving over the lane bits 16, 8, 4, 2 (a lane keeps the upper or
// lower half of its columns by that bit and takes the maximum with its
// partner's copy of the same half), then one exchange over bit 1.  Lanes 2c
// and 2c+1 return the maximum of column c over all 32 lanes.
// (col_sum16: the same pattern with additions.)
template <bool kSum>
__device__ __forceinline__ float col_reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int m = 16, n = 8; m >= 2; m >>= 1, n >>= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = upper ? v[i] : v[i + n];
            const float keep = upper ? v[i + n] : v[i];
            const float got = __shfl_xor_sync(0xffffffffu, send, m);
            v[i] = kSum ? keep + got : fmaxf(keep, got);
        }
    }
    const float got = __shfl_xor_sync(0xffffffffu, v[0], 1);
    return kSum ? v[0] + got : fmaxf(v[0], got);
}
__device__ __forceinline__ float col_max16(float (&v)[16], int lane) { return col_reduce16<false>(v, lane); }
__device__ __forceinline__ float col_sum16(float (&v)[16], int lane) { return col_reduce16<true>(v, lane); }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Two bf16 (one 32-bit word) -> two fp16 (round to nearest), exact for
// magnitudes below 65536; larger magnitudes become inf.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_half2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void set_abort(Misc* ms, uint32_t* status) {
    if (atomicExch(&ms->abort_flag, 1) == 0) atomicOr(status, LUCETREE_DEV_TIMEOUT);
}
__device__ __forceinline__ bool aborted(Misc* ms) { return *(volatile int*)&ms->abort_flag != 0; }

// KQ = 1: K held as FP8 E4M3 codes with one power-of-two exponent per token
// (the codes [128 keys][128 dims] fill a 16 KB chunk, so a 256-dim K tile is
// two chunks); the queries arrive split in two E4M3 parts (tm_q: high part,
// tm_q2: low part, both scaled by one power of two per key segment) and QK
// runs as two kind::f8f6f4 MMAs per 32-dim step into the same accumulator.
// The softmax multiplies each key's scores by its exponent and the segment's
// query scale.
template <int D, bool BF16, int RGP, int VQ, int KQ>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_ve,
                     const __grid_constant__ CUtensorMap tm_q2, const AttnLaunch L) {
    using Lay = Layout<D, RGP>;
    constexpr int kChunks = Lay::kChunks;                  // Q chunks (16-bit: 64 dims; E4M3: 2 parts x 128 dims)
    constexpr int kChunksK = KQ ? D / 128 : D / 64;        // ring chunks per K operand
    constexpr int kChunksV = D / 64;                       // ring chunks per V operand
    static_assert(!KQ || (D == 256 && BF16), "E4M3 K: head dim 256, bf16 queries");
    constexpr int kNch = Lay::kNch;
    constexpr int kNa = (kNch + kSmGroups - 1) / kSmGroups;  // column chunks per softmax warp (at most)
    constexpr int kNS = Lay::kNS;
    constexpr uint32_t kAB = BF16 ? 1u : 0u;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + Lay::kQOff;
    uint8_t* sP = smem + Lay::kPOff;
    uint8_t* sSlots = smem + Lay::kSlotOff;
    Misc* ms = reinterpret_cast<Misc*>(smem + Lay::kMiscOff);

    const lucetree_attn_args& a = L.a;
    const PlanDims& p = L.plan;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rg = blockIdx.x / p.Cg, cta = blockIdx.x % p.Cg;
    const int i0 = rg * p.rg.NPG;
    const int R_seg = (min(p.N, i0 + p.rg.NPG) - i0) * p.G;
    const int RG = p.rg.RG;

    // ---------------------------------------------------------------- set-up
    // (no global memory is read here, so it overlaps the previous kernel's
    // tail under programmatic dependent launch)
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&ms->full[i], 1);
            mbar_init(&ms->empty[i], 1);
        }
        for (int i = 0; i < kMaxSlots; ++i) {
            mbar_init(&ms->vfull[i], 1);
            mbar_init(&ms->vready[i], VQ == 0 ? kConvWarps : kSmWarps);
        }
        mbar_init(&ms->s_full, 1);
        mbar_init(&ms->s_free, kSmWarps);
        mbar_init(&ms->q_full, 1);
        mbar_init(&ms->q_empty, 1);
        mbar_init(&ms->p_full, kSmWarps);
        mbar_init(&ms->pv_done, 1);
        mbar_init(&ms->drain, 1);
        mbar_init(&ms->q_ready, kSmWarps);
        ms->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp >= 4) {
        // rows RG..RGP-1 of Q are padding: zero them once (TMA never writes them)
        const int st = threadIdx.x - 128;
        for (int idx = st; idx < kChunks * RGP * 8; idx += kSoftmaxThreads) {
            const int c = idx / (RGP * 8), r = (idx / 8) % RGP, u = idx % 8;
            if (r >= RG) *reinterpret_cast<uint4*>(sQ + c * RGP * 128 + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&ms->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_q);
        if (VQ) prefetch_tensormap(&tm_ve);
        if (KQ) prefetch_tensormap(&tm_q2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms->tmem_base;

    // inputs may come from the previous kernel on the stream: wait for it, then
    // let the merge kernel start its blocks as SMs free up (it waits for this
    // grid before reading partials).  The trigger must stay after the wait: the
    // merge kernel reads the ancestor masks, queries and tree K/V before its own
    // wait, relying on this kernel having waited for their producers first.
    pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();
    const long long nT = total_tiles(p, a.ctx_len);
    const int t0 = nT ? (int)cta_begin(cta, nT, p.Cg) : 0, t1 = nT ? (int)cta_begin(cta + 1, nT, p.Cg) : 0;
    if (t0 >= t1) {  // uniform across the CTA: nothing to do but give TMEM back
        if (warp == 1) tmem_dealloc(tmem, kTmemCols);
        return;
    }
    const uint32_t n_tiles = (uint32_t)(t1 - t0);

    if (warp < 4) {
    regs_dec<kRegsIssue>();
    if (warp == 0) {
        // ============================================================ TMA producer
        const int oob_row = a.num_pages * p.Hkv * kPage;  // first row past the pool: zero fill
        const uint64_t pol_stream = policy_evict_first();  // K/V are read once: do not keep them in L2
        uint32_t chunk = 0, vchunk = 0;
        int q_loads = 0;
        bool ok = true;
        // one operand (one tile's K or V): kChunksK / kChunksV slots of two boxes each
        auto issue = [&](bool is_v, int row0, int row1) -> bool {
            for (int c = 0; c < (is_v ? kChunksV : kChunksK); ++c) {
                const int slot = chunk % kNS;
                const bool w = mbar_wait(&ms->empty[slot], ((chunk / kNS) & 1) ^ 1);
                if (!__all_sync(0xffffffffu, w)) return false;  // lanes agree on a timeout
                if (lane == 0) {
                    uint8_t* dst = sSlots + slot * kChunkBytes;
                    uint64_t* bar = &ms->full[slot];
                    if (is_v) {
                        mbar_arrive(bar);  // this fill's phase of full[slot]; the data signal is vfull
                        bar = &ms->vfull[vchunk % kMaxSlots];
                    }
                    if (VQ && is_v) {
                        // codes of [64 keys of page c & 1][dims 128 * (c >> 1) .. +127] and the
                        // page's per-token exponents
                        const int row = (c & 1) ? row1 : row0;
                        mbar_arrive_expect_tx(bar, VCodes<VQ>::kBytes + kPage);
                        tma_load_2d_hint(dst + VCodes<VQ>::kOff, &tm_v, VCodes<VQ>::kRowBytes * (c >> 1), row, bar,
                                         pol_stream);
                        tma_load_2d_hint(ms->vexp[vchunk % kMaxSlots], &tm_ve, 0, row / kPage, bar, pol_stream);
                    } else if (is_v) {
                        // [64 keys of page c & 1][dims 128 * (c >> 1) .. +127]
                        mbar_arrive_expect_tx(bar, kChunkBytes);
                        const int row = (c & 1) ? row1 : row0, x = 128 * (c >> 1);
                        tma_load_2d_hint(dst, &tm_v, x, row, bar, pol_stream);
                        tma_load_2d_hint(dst + 8192, &tm_v, x + 64, row, bar, pol_stream);
                    } else {
                        // [128 keys: page 0 then page 1][dims 64 * c .. +63] (16-bit K), or
                        // [128 keys][dims 128 * c .. +127] (E4M3 codes: x counts bytes)
                        mbar_arrive_expect_tx(bar, kChunkBytes);
                        tma_load_2d_hint(dst, &tm_k, (KQ ? 128 : 64) * c, row0, bar, pol_stream);
                        tma_load_2d_hint(dst + 8192, &tm_k, (KQ ? 128 : 64) * c, row1, bar, pol_stream);
                    }
                }
                __syncwarp();
                ++chunk;
                vchunk += is_v ? 1u : 0u;
            }
            return true;
        };
        TileCursor cur;
        cur.start(t0, t1, p, a.ctx_len);
        int npages = 0;
        const int32_t* pt = a.page_table;
        // page ids of the current piece, 16 tiles (32 pages) per warp-wide load, one batch ahead
        auto load_batch = [&](int tb) {
            const int pg = 2 * tb + lane;
            int pid = -1;
            if (pg < npages && pg < 2 * cur.pc.te) {
                const int v = pt[pg];
                if (v >= 0 && v < a.num_pages) pid = v;
                else atomicOr(a.status, LUCETREE_DEV_BAD_PAGE);
            }
            return pid;
        };
        int pid_cur = -1, pid_next = -1;
        int v_row0 = 0, v_row1 = 0;
        bool have_v = false;
        while (ok && cur.live) {
            const int rel = cur.t - cur.pc.ta;
            if (rel == 0) {
                // a new key segment: its queries replace the previous ones once their last QK is done
                if (KQ && cur.piece_no > 0 && have_v) {
                    // E4M3 K: the previous piece's last V goes first, because the next
                    // piece's first QK waits for the softmax warps to split its queries,
                    // which they do only after that V's PV (the MMA warp keeps this order)
                    if (!(ok = issue(true, v_row0, v_row1))) break;
                    have_v = false;
                }
                if (cur.piece_no > 0) {
                    const bool w = mbar_wait(&ms->q_empty, (cur.piece_no - 1) & 1);
                    if (!(ok = __all_sync(0xffffffffu, w))) break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&ms->q_full, kChunks * RG * 128);
                    const int b = cur.pc.s / p.Hkv, g = cur.pc.s % p.Hkv;
                    // (E4M3 K: the bf16 queries too; the softmax warps split them in place)
                    for (int c = 0; c < kChunks; ++c)
                        tma_load_3d(sQ + c * RGP * 128, &tm_q, 64 * c, g * p.G, b * p.N + i0, &ms->q_full);
                }
                __syncwarp();
                ++q_loads;
                npages = (cur.pc.L + kPage - 1) / kPage;
                pt = a.page_table + (size_t)(cur.pc.s / p.Hkv) * p.max_pages;
                pid_cur = load_batch(cur.pc.ta);
                pid_next = load_batch(cur.pc.ta + 16);
            } else if ((rel & 15) == 0) {
                pid_cur = pid_next;
                pid_next = load_batch(cur.t + 16);
            }
            int row[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pid = __shfl_sync(0xffffffffu, pid_cur, 2 * (rel & 15) + h);
                row[h] = pid >= 0 ? (pid * p.Hkv + cur.pc.s % p.Hkv) * kPage : oob_row;
            }
            if (!(ok = issue(false, row[0], row[1]))) break;
            if (have_v && !(ok = issue(true, v_row0, v_row1))) break;
            v_row0 = row[0];
            v_row1 = row[1];
            have_v = true;
            cur.step(p, a.ctx_len);
        }
        if (ok && have_v) ok = issue(true, v_row0, v_row1);
        if (!ok || aborted(ms)) {
            set_abort(ms, a.status);
            // wait (bounded) for this CTA's own copies still in flight
            if (lane == 0) {
                // (full[] covers the K fills, vfull[] the V fills; each wait on a
                // barrier whose phase already completed returns at once)
                const uint32_t first = chunk > (uint32_t)kNS ? chunk - kNS : 0u;
                for (uint32_t c = first; c < chunk; ++c) mbar_wait(&ms->full[c % kNS], (c / kNS) & 1, 200000000ll);
                const uint32_t vfirst = vchunk > (uint32_t)kNS ? vchunk - kNS : 0u;
                for (uint32_t c = vfirst; c < vchunk; ++c)
                    mbar_wait(&ms->vfull[c % kMaxSlots], (c / kMaxSlots) & 1, 200000000ll);
                if (q_loads > 0) mbar_wait(&ms->q_full, (q_loads - 1) & 1, 200000000ll);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            // (for E4M3 K the same descriptor bits read as E4M3 x E4M3 under kind::f8f6f4)
            const uint32_t id_qk = idesc_f16(128, RGP, KQ ? 0u : kAB, 0, 0);
            const uint32_t id_pv = idesc_f16(128, RGP, 0u, 1, 1);  // fp16 V and P
            constexpr uint64_t hi_k = desc_hi(16, 1024, kLayoutSwizzle128);
            constexpr uint64_t hi_v = desc_hi(8192, 1024, kLayoutSwizzle128);  // 2nd 64-dim box at +8 KB
            constexpr uint64_t hi_p = desc_hi(128, 2048, kLayoutInterleave);
            const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP), aS = smem_u32(sSlots);
            uint32_t chunk = 0, jq = 0, j = 0;
            bool ok = true;
            TileCursor qk, pv;
            qk.start(t0, t1, p, a.ctx_len);
            pv.start(t0, t1, p, a.ctx_len);
            // S^T(jq) = K(jq) . Q^T; S^T is free once the softmax has read tile jq-1
            auto issue_qk = [&]() -> bool {
                if (jq > 0) {
                    if (!mbar_wait(&ms->s_free, (jq - 1) & 1)) return false;
                    tc_fence_after();
                }
                if (qk.first()) {
                    if (!mbar_wait(KQ ? &ms->q_ready : &ms->q_full, qk.piece_no & 1)) return false;
                    tc_fence_after();
                }
                for (int c = 0; c < kChunksK; ++c) {
                    const int slot = chunk % kNS;
                    if (!mbar_wait(&ms->full[slot], (chunk / kNS) & 1)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        const uint64_t ad = make_desc(hi_k, aS + slot * kChunkBytes + sub * 32);
                        if constexpr (KQ) {
                            // 32 dims per step (dims 128 c + 32 sub): K codes times the high,
                            // then the low query part; the split queries keep each 32-dim
                            // span's hi codes in the first 32 bytes of the span's 64 and lo
                            // in the next 32, the spans at the bf16 layout's places
                            const uint32_t qspan = aQ + (2 * c + (sub >> 1)) * RGP * 128 + (sub & 1) * 64;
                            const uint64_t bh = make_desc(hi_k, qspan);
                            const uint64_t bl = make_desc(hi_k, qspan + 32);
                            mma_f8f6f4_ss(tmem, ad, bh, id_qk, (c | sub) != 0);
                            mma_f8f6f4_ss(tmem, ad, bl, id_qk, 1u);
                        } else {
                            const uint64_t bd = make_desc(hi_k, aQ + c * RGP * 128 + sub * 32);
                            mma_f16_ss(tmem, ad, bd, id_qk, (c | sub) != 0);
                        }
                    }
                    mma_commit(&ms->empty[slot]);
                    ++chunk;
                }
                mma_commit(&ms->s_full);
                if (qk.last()) mma_commit(&ms->q_empty);
                ++jq;
                qk.step(p, a.ctx_len);
                return true;
            };
            if (qk.live) ok = issue_qk();
            while (ok && pv.live) {
                if (aborted(ms)) {
                    ok = false;
                    break;
                }
                // QK(j+1), then PV(j); with E4M3 K, QK(j+1) after PV(j) when it opens a
                // new piece (its queries are split by the softmax warps once they are
                // done with tile j).  One loop over the two steps keeps a single copy
                // of each in this 56-register warp.
                const bool defer_qk = KQ && qk.live && qk.first() && qk.piece_no > 0;
#pragma unroll 1
                for (int step = 0; step < 2 && ok; ++step) {
                    if ((step == 0) != defer_qk) {
                        if (qk.live) ok = issue_qk();
                        continue;
                    }
                    // O^T += V^T . P^T once the softmax has written P^T(j)
                    if (!(ok = mbar_wait(&ms->p_full, j & 1))) break;
                    tc_fence_after();
                    const bool first = pv.first();
                    // output dims 128h..128h+127: chunk 2h holds keys 0..63, chunk
                    // 2h+1 keys 64..127 (four 16-key steps each)
                    for (int h = 0; h < kChunksV / 2 && ok; ++h) {
                        const uint32_t dO = tmem + (h ? Lay::kColO1 : Lay::kColO0);
                        for (int kh = 0; kh < 2 && ok; ++kh) {
                            const int slot = chunk % kNS;
                            // landed and made the fp16 operand
                            const uint32_t vn = j * kChunksV + 2 * h + kh;
                            if (!(ok = mbar_wait(&ms->vready[vn % kMaxSlots], (vn / kMaxSlots) & 1))) break;
                            tc_fence_after();
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks) {
                                const uint64_t ad = make_desc(hi_v, aS + slot * kChunkBytes + ks * 2048);
                                const uint64_t bd = make_desc(hi_p, aP + (4 * kh + ks) * 256);
                                mma_f16_ss(dO, ad, bd, id_pv, !(first && kh == 0 && ks == 0));
                            }
                            mma_commit(&ms->empty[slot]);
                            ++chunk;
                        }
                    }
                    if (!ok) break;
                    mma_commit(&ms->pv_done);
                    ++j;
                    pv.step(p, a.ctx_len);
                }
            }
            if (!ok || aborted(ms)) {
                set_abort(ms, a.status);
                mma_commit(&ms->drain);  // every MMA issued so far has finished before TMEM is freed
                mbar_wait(&ms->drain, 0, 200000000ll);
            }
        }
        __syncwarp();
    } else if (VQ == 0) {
        // ============================================================ V conversion (warps 2, 3)
        // Each 16-bit V chunk, once landed: bf16 -> fp16 in place (exact below
        // 65536; a larger magnitude becomes inf and the merge flags the row),
        // and the rows of keys at or past L in a partial page zeroed (the pool
        // holds arbitrary data there and 0 * NaN would poison O^T); then
        // vready.  Doing this here rather than in the softmax warps keeps a
        // late V tile from holding up the next tile's exponents.  Thread ct
        // owns 16-byte units ct + 64 i of a chunk; unit u holds 8 dims of key
        // 64 * (c & 1) + (u % 512) / 8 (each 8 KB box is [64 keys][128 B]; the
        // swizzle permutes units only within a key's row).
        const int ct = threadIdx.x - 64;  // 0 .. 63
        TileCursor cur;
        cur.start(t0, t1, p, a.ctx_len);
        uint32_t j = 0;
        bool ok = true;
        while (ok && cur.live) {
            const int nvalid = min(kTileKeys, cur.pc.L - cur.t * kTileKeys);
            // ring position of V(j)'s first chunk: the K operands before it
            // (K(0) .. K(j+1), or .. K(j) for the last tile) and V(0) .. V(j-1)
            // (E4M3 K: the next piece's first K comes after this V)
            const bool k_after = j + 1 < n_tiles && !(KQ && cur.t == cur.pc.te - 1);
            const uint32_t vbase = (k_after ? j + 2 : j + 1) * kChunksK + j * kChunksV;
            for (int c = 0; c < kChunksV; ++c) {
                const uint32_t vn = j * kChunksV + c;
                const bool landed = mbar_wait(&ms->vfull[vn % kMaxSlots], (vn / kMaxSlots) & 1);
                if (!__all_sync(0xffffffffu, landed) || aborted(ms)) {
                    ok = false;
                    break;
                }
                uint4* base = reinterpret_cast<uint4*>(sSlots + ((vbase + c) % kNS) * kChunkBytes);
                const int nv = nvalid - 64 * (c & 1);  // valid keys of this chunk's page
                constexpr int kUnits = kChunkBytes / 16 / (32 * kConvWarps);  // 16 per thread
                constexpr int kBatch = 4;                                      // loads in flight
                if (BF16 && nv >= 64) {
                    // a full page (every chunk but a segment's last few): no per-key test
#pragma unroll 1
                    for (int i0 = 0; i0 < kUnits; i0 += kBatch) {
                        uint4 x[kBatch];
#pragma unroll
                        for (int k = 0; k < kBatch; ++k) x[k] = base[ct + 32 * kConvWarps * (i0 + k)];
#pragma unroll
                        for (int k = 0; k < kBatch; ++k) {
                            x[k].x = bf16x2_to_f16x2(x[k].x);
                            x[k].y = bf16x2_to_f16x2(x[k].y);
                            x[k].z = bf16x2_to_f16x2(x[k].z);
                            x[k].w = bf16x2_to_f16x2(x[k].w);
                            base[ct + 32 * kConvWarps * (i0 + k)] = x[k];
                        }
                    }
                } else if (BF16 || nv < 64) {
#pragma unroll 1
                    for (int i0 = 0; i0 < kUnits; i0 += kBatch) {
                        uint4 x[kBatch];
                        bool kv[kBatch];
#pragma unroll
                        for (int k = 0; k < kBatch; ++k) {
                            const int u = ct + 32 * kConvWarps * (i0 + k);
                            kv[k] = ((u & 511) >> 3) < nv;
                            x[k] = kv[k] ? base[u] : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int k = 0; k < kBatch; ++k) {
                            const int u = ct + 32 * kConvWarps * (i0 + k);
                            if constexpr (BF16) {
                                x[k].x = bf16x2_to_f16x2(x[k].x);
                                x[k].y = bf16x2_to_f16x2(x[k].y);
                                x[k].z = bf16x2_to_f16x2(x[k].z);
                                x[k].w = bf16x2_to_f16x2(x[k].w);
                            }
                            if (BF16 || !kv[k]) base[u] = x[k];
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms->vready[vn % kMaxSlots]);
            }
            ++j;
            cur.step(p, a.ctx_len);
        }
        if (!ok) set_abort(ms, a.status);
    }
    } else {
        regs_inc<kRegsSoftmax>();
        // ============================================================ softmax + epilogue
        // 12 warps: warp w reads TMEM lanes 32*(w%4)..+31 (its key lanes) and
        // handles share hf = (w-4)/4 of the row tile's column chunks.
        const int quarter = warp & 3;
        const int hf = (warp - 4) >> 2;
        const int kl = quarter * 32 + lane;  // key lane of S^T, output dim of O^T
        const int st = threadIdx.x - 128;    // 0..383
        const int cb = min(hf * kNa, kNch), ce = min(cb + kNa, kNch);
        const int nch = ce - cb;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        float sl2 = L.scale_log2;  // E4M3 K: set per tile from the key's exponent and the segment's query scale
        const int my_half = kl >> 6;  // which 64-token page of the tile holds my key
        uint32_t j = 0;
        bool bad = false;  // warp-uniform at every tcgen05 load / store below
        // bounded wait whose outcome all lanes of the warp agree on
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            const bool w = mbar_wait(bar, parity);
            return __all_sync(0xffffffffu, w);
        };
        // One streaming pass over my chunks of S^T: P = 2^(s*scale*log2e - m)
        // with the current shifts; lpart += P (sign +1) or -= P (sign -1, the
        // exact undo of a pass made with the same shifts); optionally keeps
        // P (fp16 pairs) in registers `ph` and tracks the largest exponent.
        // Invalid keys and padding columns give P = 0.
        // P stays in registers so that the pass can run while PV of the
        // previous tile still reads the shared P^T buffer; store_p writes it
        // once that PV has completed.
        auto exp_pass = [&](float (&lpart)[kNa * 16], bool valid, float sign, bool keep_p, float& ex,
                            uint32_t (&ph)[kNa * 8]) {
            // 16-column chunks, each in two 8-column blocks b = 2*cc + hb; the
            // TMEM load of chunk cc+1 is in flight while chunk cc is computed.
            // An invalid key's exponents are -inf, and so are a padding
            // column's (its shift is +inf), so neither needs a column test.
            uint32_t rn[16];
            tmem_ld16(tl + 16 * cb, rn);
#pragma unroll
            for (int cc = 0; cc < kNa; ++cc) {
                if (cc >= nch) continue;
                uint32_t r[16];
                tmem_wait_ld_regs16(rn);
#pragma unroll
                for (int k = 0; k < 16; ++k) r[k] = rn[k];
                if (cc + 1 < nch) tmem_ld16(tl + 16 * (cb + cc + 1), rn);
                const int c = cb + cc;
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    const int bi = 2 * cc + hb;
                    const float4* m4 = reinterpret_cast<const float4*>(ms->m_ref + 16 * c + 8 * hb);
                    const float4 ma = m4[0], mb = m4[1];
                    const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
                    float pv[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float x = valid ? fmaf(__uint_as_float(r[8 * hb + k]), sl2, -mv[k]) : -INFINITY;
                        ex = fmaxf(ex, x);
                        pv[k] = ex2(x);
                        float& acc = lpart[cc * 16 + 8 * hb + k];
                        acc = fmaf(sign, pv[k], acc);
                    }
                    if (keep_p) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) ph[4 * bi + k] = pack_half2(pv[2 * k], pv[2 * k + 1]);
                    }
                }
            }
        };
        // P^T [8-column block][128 keys][8 columns] fp16: block 2c + hb of my chunks
        auto store_p = [&](const uint32_t (&ph)[kNa * 8]) {
#pragma unroll
            for (int bi = 0; bi < 2 * kNa; ++bi) {
                if (bi >= 2 * nch) continue;
                const int nb = 2 * cb + bi;
                *reinterpret_cast<uint4*>(sP + nb * 2048 + kl * 16) =
                    make_uint4(ph[4 * bi], ph[4 * bi + 1], ph[4 * bi + 2], ph[4 * bi + 3]);
            }
        };

        TileCursor cur;
        cur.start(t0, t1, p, a.ctx_len);

        while (cur.live) {
            const int piece_no = cur.piece_no;
            const int seg = cur.pc.s;
            bar_sync(1, kSoftmaxThreads);
            // padding columns keep a shift of +inf, so their exponents are -inf and P = 0
            for (int col = st; col < RGP; col += kSoftmaxThreads) ms->m_ref[col] = col < R_seg ? -INFINITY : INFINITY;
            bar_sync(1, kSoftmaxThreads);
            float lpart[kNa * 16];
#pragma unroll
            for (int i = 0; i < kNa * 16; ++i) lpart[i] = 0.f;
            uint32_t page_bits = 0;
            int pid_lane = -1;  // E4M3 K: page id of my key's page for tile (batch start + lane)
            // E4M3 K: my key's exponent byte, loaded one tile ahead; the segment's query scale
            auto page_of = [&](int tile) -> int {
                const int pg = 2 * tile + my_half;
                return pg < (cur.pc.L + kPage - 1) / kPage ? a.page_table[(size_t)(seg / p.Hkv) * p.max_pages + pg] : -1;
            };
            auto k_exp_of = [&](int pid) -> uint32_t {
                return pid >= 0 && pid < a.num_pages
                           ? (uint32_t)L.k_exp[((size_t)pid * p.Hkv + seg % p.Hkv) * kPage + (kl & (kPage - 1))]
                           : 0u;
            };
            uint32_t ek_next = 0;
            float qs = 0.f;
            int pg0 = -1;  // E4M3 K: my key's page for the piece's first tile (its exponent is read after the split)
            if constexpr (KQ) {
                pg0 = page_of(cur.pc.ta);
                // The piece's bf16 queries (four 64-dim chunks of [RGP rows][128 B],
                // 128-byte swizzled) become two E4M3 parts in place, scaled by 2^p so
                // that their largest magnitude lies in (224, 448]: hi = e4m3(q 2^p),
                // lo = e4m3(q 2^p - hi).  The 64 bytes of each 32-dim span of a row
                // (four 16-byte units) are rewritten as hi's 32 codes in the first
                // two units and lo's in the last two, so every thread rewrites only
                // what it read, and a 32-dim K step of the FP8 MMA finds its hi (and,
                // 32 bytes on, its lo) operand rows contiguous.  One pass for the
                // CTA's largest |q| (one barrier, which also carries a timed-out
                // wait), one to convert.
                constexpr int kSpans = RGP * 8;
                constexpr int kPer = (kSpans + kSoftmaxThreads - 1) / kSoftmaxThreads;
                const bool qw = !bad && wait_all(&ms->q_full, piece_no & 1);
                auto span_unit = [&](int sid, int k) -> uint4* {
                    const int r = sid >> 3, v = sid & 7;
                    return reinterpret_cast<uint4*>(sQ + (v >> 1) * RGP * 128 + r * 128 +
                                                    (((4 * (v & 1) + k) ^ (r & 7)) << 4));
                };
                float qm = 0.f;
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const int sid = st + kSoftmaxThreads * i;
                    if (sid >= kSpans || !qw) continue;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float v[8];
                        const uint4 w4 = *span_unit(sid, k);
                        load8_f32<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(&w4), v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) qm = fmaxf(qm, fabsf(v[e]));
                    }
                }
                qm = warp_max(qm);
                if (lane == 0) ms->col_red[0][warp - 4] = qm;
                if (bar_sync_or(1, kSoftmaxThreads, !qw)) bad = true;
                if (!bad) {
                    qm = 0.f;
#pragma unroll
                    for (int w = 0; w < kSmWarps; ++w) qm = fmaxf(qm, ms->col_red[0][w]);
                    const int pe = e4m3::scale_exponent(qm);
                    qs = ldexpf(L.scale_log2, -pe);
                    const float s2p = ldexpf(1.f, pe);  // 2^p: scaling by it is exact here
#pragma unroll
                    for (int i = 0; i < kPer; ++i) {
                        const int sid = st + kSoftmaxThreads * i;
                        if (sid >= kSpans) continue;
                        uint4 w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) w4[k] = *span_unit(sid, k);
                        uint32_t hw[8], lw[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            float v[8];
                            load8_f32<__nv_bfloat16>(reinterpret_cast<const __nv_bfloat16*>(&w4[k]), v);
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float y0 = v[e] * s2p, y1 = v[e + 1] * s2p;  // exact: |y| <= 448
                                const uint16_t hc = e4m3::e4m3x2(y0, y1);
                                const float2 hf = e4m3::e4m3x2_to_f32(hc);
                                const uint16_t lc = e4m3::e4m3x2(y0 - hf.x, y1 - hf.y);  // exact differences
                                const int wi = 2 * k + (e >> 2);  // dims 8k + e, 8k + e + 1
                                if ((e & 2) == 0) {
                                    hw[wi] = hc;
                                    lw[wi] = lc;
                                } else {
                                    hw[wi] |= (uint32_t)hc << 16;
                                    lw[wi] |= (uint32_t)lc << 16;
                                }
                            }
                        }
                        *span_unit(sid, 0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *span_unit(sid, 1) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                        *span_unit(sid, 2) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        *span_unit(sid, 3) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ms->q_ready);
                }
            }

            if constexpr (KQ) ek_next = k_exp_of(pg0);
            while (cur.live && cur.piece_no == piece_no) {
                const int t = cur.t;
                // validity of my page for 32 tiles at a time (one load per lane)
                const int tb = (t - cur.pc.ta) & 31;
                if (tb == 0) {
                    const int tt = t + lane;
                    const int pg = 2 * tt + my_half;
                    bool okp = false;
                    pid_lane = -1;
                    if (tt < cur.pc.te && pg < (cur.pc.L + kPage - 1) / kPage) {
                        const int pid = a.page_table[(size_t)(seg / p.Hkv) * p.max_pages + pg];
                        okp = pid >= 0 && pid < a.num_pages;
                        pid_lane = pid;
                    }
                    page_bits = __ballot_sync(0xffffffffu, okp);
                }
                const int nvalid = min(kTileKeys, cur.pc.L - t * kTileKeys);
                const bool page_ok = (page_bits >> tb) & 1u;
                const bool valid = kl < nvalid && page_ok;
                const bool first = cur.first();
                if constexpr (KQ) {
                    // this tile's exponent was loaded during the previous tile; load the next one's
                    const uint32_t ek = valid ? ek_next : 0u;
                    if (t + 1 < cur.pc.te) {
                        const int pid1 = tb + 1 < 32 ? __shfl_sync(0xffffffffu, pid_lane, tb + 1) : page_of(t + 1);
                        ek_next = k_exp_of(pid1);
                    }
                    sl2 = qs * __uint_as_float(ek << 23);  // x 2^(e - 127); e = 0 reads as zero
                }

                // S^T(j) ready (P^T and O^T are waited for later: PV(j-1) may still
                // be reading P^T while this tile's exponents are computed)
                if (!bad && !wait_all(&ms->s_full, j & 1)) bad = true;
                if (!bad) tc_fence_after();
                bool pv_prev_done = j == 0;  // PV(j-1) known complete

                // pass 0: exponents with the current shifts (P kept in registers,
                //         sums added, largest exponent voted across the CTA)
                // pass 1: if an exponent exceeded kTau, the same pass with the sums
                //         subtracted (exact undo)
                // pass 2: exact column maxima move the shifts, then P and sums again
                // The first tile of a range has no shifts yet and starts at pass 2.
                float ex = -INFINITY;
                uint32_t ph[kNa * 8];
                if (!bad && !first) {
                    exp_pass(lpart, valid, 1.f, true, ex, ph);
                }
                // one barrier decides the path; a second one only when it says
                // "slow", to tell a timeout (somewhere) from a shift update
                const bool bad_now = bad || aborted(ms);
                const bool slow = bar_sync_or(1, kSoftmaxThreads, bad_now || first || ex > kTau);
                if (slow && bar_sync_or(1, kSoftmaxThreads, bad_now)) {
                    bad = true;
                    break;
                }
                if (slow) {
                    if (!first) exp_pass(lpart, valid, -1.f, false, ex, ph);  // pass 1
                    // pass 2: exact column maxima of this tile, then move the shifts
#pragma unroll 1
                    for (int cc = 0; cc < nch; ++cc) {
                        const int c = cb + cc;
                        uint32_t r[16];
                        tmem_ld16(tl + 16 * c, r);
                        tmem_wait_ld_regs16(r);
                        const int lim = valid ? R_seg - 16 * c : 0;
                        float v[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = k < lim ? __uint_as_float(r[k]) * sl2 : -INFINITY;
                        // maxima of the 16 columns over the warp's 32 key lanes
                        const float cm = col_max16(v, lane);
                        if ((lane & 1) == 0) ms->col_red[quarter][16 * c + (lane >> 1)] = cm;
                    }
                    bar_sync(1, kSoftmaxThreads);
                    for (int col = st; col < RGP; col += kSoftmaxThreads) {
                        const float cm = fmaxf(fmaxf(ms->col_red[0][col], ms->col_red[1][col]),
                                               fmaxf(ms->col_red[2][col], ms->col_red[3][col]));
                        const float mo = ms->m_ref[col];
                        const float mn = fmaxf(mo, cm);
                        ms->alpha[col] = mn > mo ? ex2(mo - mn) : 1.f;
                        ms->m_ref[col] = mn;
                    }
                    bar_sync(1, kSoftmaxThreads);
#pragma unroll
                    for (int cc = 0; cc < kNa; ++cc) {
                        if (cc >= nch) continue;
#pragma unroll
                        for (int k = 0; k < 16; ++k) lpart[cc * 16 + k] *= ms->alpha[16 * (cb + cc) + k];
                    }
                    if (!first) {
                        // O^T columns accumulated so far move with their shift, once
                        // PV(j-1) has finished adding to them (a warp that timed out
                        // here skips its TMEM accesses but keeps to the barriers)
                        if (!bad && j > 0 && !wait_all(&ms->pv_done, (j - 1) & 1)) bad = true;
                        pv_prev_done = true;
                        if (!bad) tc_fence_after();
#pragma unroll 1
                        for (int cc = 0; cc < nch && !bad; ++cc) {
                            const int c = cb + cc;
                            bool any = false;
#pragma unroll
                            for (int k = 0; k < 16; ++k) any |= ms->alpha[16 * c + k] != 1.f;
                            if (!any) continue;
#pragma unroll 1
                            for (int h = 0; h < Lay::kDh; ++h) {
                                uint32_t r[16];
                                const uint32_t addr = tl + (h ? Lay::kColO1 : Lay::kColO0) + 16 * c;
                                tmem_ld16(addr, r);
                                tmem_wait_ld_regs16(r);
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    r[k] = __float_as_uint(__uint_as_float(r[k]) * ms->alpha[16 * c + k]);
                                tmem_st16(addr, r);
                            }
                        }
                        if (!bad) tmem_wait_st();
                    }
                    if (!bad) exp_pass(lpart, valid, 1.f, true, ex, ph);
                }
                // S^T is no longer read: the next tile's QK may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ms->s_free);

                // P^T is free once PV(j-1) has completed; then this tile's P goes in
                if (!bad && !pv_prev_done && !wait_all(&ms->pv_done, (j - 1) & 1)) bad = true;
                if (!bad) {
                    tc_fence_after();
                    store_p(ph);
                }
                tc_fence_before();
                fence_proxy_async_smem();  // P^T stores -> tensor-core reads
                __syncwarp();              // every lane's stores and fence come before lane 0's arrive
                if (!bad && lane == 0) mbar_arrive(&ms->p_full);

                // Quantised V(j), chunk by chunk as it lands: the codes expanded in
                // place to the fp16 operand, rows of keys at or past L zeroed (the
                // pool holds arbitrary data there and 0 * NaN would poison O^T).
                // (16-bit V is converted by warps 2 and 3.)  Unit u of a chunk holds
                // 8 dims of key 64 * (c & 1) + (u % 512) / 8 (each 8 KB box is
                // [64 keys][128 B]; the swizzle permutes units only within a key's row).
                if (!bad && VQ != 0) {
                    // ring position of V(j)'s first chunk: the K operands before it
                    // (K(0) .. K(j+1), or .. K(j) for the last tile) and V(0) .. V(j-1)
                    const bool k_after = j + 1 < n_tiles && !(KQ && t == cur.pc.te - 1);
                    const uint32_t vbase = (k_after ? j + 2 : j + 1) * kChunksK + j * kChunksV;
                    for (int c = 0; c < kChunksV; ++c) {
                        const uint32_t vn = j * kChunksV + c;
                        const bool landed = wait_all(&ms->vfull[vn % kMaxSlots], (vn / kMaxSlots) & 1);
                        if (VQ != 2 && !landed) {  // (int4 reports a timeout through its barrier)
                            bad = true;
                            break;
                        }
                        uint4* base = reinterpret_cast<uint4*>(sSlots + ((vbase + c) % kNS) * kChunkBytes);
                        const int nv = nvalid - 64 * (c & 1);  // valid keys of this chunk's page
                        if constexpr (VQ == 1) {
                            // int8: the fp16 output of key row r covers bytes [128 r, 128 r + 128) of
                            // each 8 KB box; the second box's lands exactly on row r's own 128 code
                            // bytes and nowhere else.  So one half-warp expands one row (lane l of
                            // 16: box l / 8, swizzled unit l % 8), its three rows' codes all read
                            // before any write: a __syncwarp suffices, no CTA barrier.  Both halves of a warp
                            // always get the same number of rows (rows hw, hw + 24, hw + 48).
                            const uint8_t* codes = reinterpret_cast<const uint8_t*>(base) + VCodes<1>::kOff;
                            const uint8_t* ex = ms->vexp[vn % kMaxSlots];
                            const int hw = 2 * (warp - 4) + (lane >> 4), l = lane & 15;
                            uint2 cws[3];
                            uint32_t ebs[3];
#pragma unroll
                            for (int it = 0; it < 3; ++it) {  // every row's codes read before any write
                                const int r = hw + 24 * it;
                                const int d0 = 64 * (l >> 3) + 8 * ((l & 7) ^ (r & 7));
                                cws[it] = make_uint2(0, 0);
                                ebs[it] = 0;
                                if (r < 64 && r < nv) {
                                    cws[it] = *reinterpret_cast<const uint2*>(codes + r * 128 + d0);
                                    ebs[it] = ex[r];
                                }
                            }
                            __syncwarp();
#pragma unroll
                            for (int it = 0; it < 3; ++it) {
                                const int r = hw + 24 * it;
                                const int u = (l >> 3) * 512 + r * 8 + (l & 7);
                                const uint2 cw = cws[it];
                                const uint32_t eb = ebs[it];
                                if (r < 64) {
                                    const float sc = __uint_as_float(eb << 23);  // 2^(e - 127)
                                    // (with E4M3 K the fp32 route below measured faster in this kernel)
                                    if (!KQ && eb >= 103 && eb <= 132) {
                                        // 2^(e-127) and 1152 * 2^(e-127) are fp16 numbers: each code c
                                        // becomes the fp16 1024 + (c + 128) (its byte under an exponent
                                        // of 2^10), and one fused (x - 1152) * 2^(e-127) per pair is exact
                                        const uint32_t s2 = pack_half2(sc, sc), n2 = pack_half2(-1152.f * sc, -1152.f * sc);
                                        const uint32_t ux = cw.x ^ 0x80808080u, uy = cw.y ^ 0x80808080u;
                                        base[u] = make_uint4(hfma2(prmt(ux, 0x64646464u, 0x5140u), s2, n2),
                                                             hfma2(prmt(ux, 0x64646464u, 0x5342u), s2, n2),
                                                             hfma2(prmt(uy, 0x64646464u, 0x5140u), s2, n2),
                                                             hfma2(prmt(uy, 0x64646464u, 0x5342u), s2, n2));
                                    } else {
                                        float f[8];
#pragma unroll
                                        for (int e = 0; e < 8; ++e)
                                            f[e] = (float)(int)(int8_t)(((e < 4 ? cw.x : cw.y) >> (8 * (e & 3))) & 0xFFu) * sc;
                                        base[u] = make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]),
                                                             pack_half2(f[4], f[5]), pack_half2(f[6], f[7]));
                                    }
                                }
                            }
                        } else if constexpr (VQ == 2) {
                            // output unit u: box u / 512 (dims 64 * box ..), key row r, 16-byte unit
                            // p of the swizzled row = logical 8-dim group p ^ (r % 8); its codes
                            // are read for every unit first, since the fp16 output overwrites them
                            const uint8_t* codes = reinterpret_cast<const uint8_t*>(base) + VCodes<VQ>::kOff;
                            const uint8_t* ex = ms->vexp[vn % kMaxSlots];
                            uint2 cw[3];
                            uint32_t eb[3];
#pragma unroll
                            for (int i = 0; i < 3; ++i) {
                                const int u = st + kSoftmaxThreads * i;
                                cw[i] = make_uint2(0, 0);
                                eb[i] = 0;
                                if (landed && u < 1024) {
                                    const int r = (u & 511) >> 3, d0 = 64 * (u >> 9) + 8 * ((u & 7) ^ (r & 7));
                                    if (r < nv) {
                                        if constexpr (VQ == 1)
                                            cw[i] = *reinterpret_cast<const uint2*>(codes + r * 128 + d0);
                                        else
                                            cw[i].x = *reinterpret_cast<const uint32_t*>(codes + r * 64 + d0 / 2);
                                        eb[i] = ex[r];
                                    }
                                }
                            }
                            // every softmax warp arrives, also after a timed-out wait: the OR
                            // tells all of them to leave together
                            if (bar_sync_or(1, kSoftmaxThreads, !landed)) {
                                bad = true;
                                break;
                            }
#pragma unroll
                            for (int i = 0; i < 3; ++i) {
                                const int u = st + kSoftmaxThreads * i;
                                if (u < 1024) {
                                    const float sc = __uint_as_float(eb[i] << 23);  // 2^(e - 127)
                                    if (eb[i] >= 103 && eb[i] <= 132) {
                                        // as for int8: nibbles with their sign bit flipped (c + 8) go
                                        // into bytes in dimension order, each byte under an fp16
                                        // exponent of 2^10, then one exact fused (x - 1032) * 2^(e-127)
                                        const uint32_t s2 = pack_half2(sc, sc), n2 = pack_half2(-1032.f * sc, -1032.f * sc);
                                        const uint32_t w = cw[i].x ^ 0x88888888u;
                                        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
                                        const uint32_t p0 = prmt(lo, hi, 0x5140u), p1 = prmt(lo, hi, 0x7362u);
                                        base[u] = make_uint4(hfma2(prmt(p0, 0x64646464u, 0x5140u), s2, n2),
                                                             hfma2(prmt(p0, 0x64646464u, 0x5342u), s2, n2),
                                                             hfma2(prmt(p1, 0x64646464u, 0x5140u), s2, n2),
                                                             hfma2(prmt(p1, 0x64646464u, 0x5342u), s2, n2));
                                    } else {
                                        float f[8];
#pragma unroll
                                        for (int e = 0; e < 8; ++e) f[e] = (float)(((int)(cw[i].x << (28 - 4 * e))) >> 28) * sc;
                                        base[u] = make_uint4(pack_half2(f[0], f[1]), pack_half2(f[2], f[3]),
                                                             pack_half2(f[4], f[5]), pack_half2(f[6], f[7]));
                                    }
                                }
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ms->vready[vn % kMaxSlots]);
                    }
                }
                ++j;
                cur.step(p, a.ctx_len);
            }

            // ---------------------------------------------------------- epilogue
            // Row sums and shifts first: they are final once the last tile's
            // exponent pass is done, so they are written while the last PV
            // (which waits for the last V tile to land) is still running.
            // Row sums: the warp's 32 key lanes by a butterfly reduce-scatter,
            // then the four lane quarters through shared memory.
#pragma unroll
            for (int cc = 0; cc < kNa; ++cc) {
                if (cc >= nch) continue;
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = lpart[cc * 16 + k];
                const float cs = col_sum16(v, lane);
                if ((lane & 1) == 0) ms->col_red[quarter][16 * (cb + cc) + (lane >> 1)] = cs;
            }
            bar_sync(1, kSoftmaxThreads);
            float* slot = L.ws + slot_index(p, rg, cta, seg) * slot_floats(p);
            float* slot_m = slot + (size_t)RG * D;
            float* slot_l = slot_m + RG;
            for (int col = st; col < R_seg; col += kSoftmaxThreads) {
                slot_l[col] = (ms->col_red[0][col] + ms->col_red[1][col]) + (ms->col_red[2][col] + ms->col_red[3][col]);
                slot_m[col] = ms->m_ref[col];
            }
            // the consensus point for a timeout in the piece's last tile (a
            // piece that failed has written garbage sums; the call reports the
            // failure through the status word)
            const bool got = !bad && mbar_wait(&ms->pv_done, (j - 1) & 1);
            if (bar_sync_or(1, kSoftmaxThreads, bad || !got || aborted(ms))) {
                bad = true;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < kNa; ++cc) {
                if (cc >= nch) continue;
                const int c = cb + cc;
#pragma unroll
                for (int h = 0; h < Lay::kDh; ++h) {
                    uint32_t r[16];
                    tmem_ld16(tl + (h ? Lay::kColO1 : Lay::kColO0) + 16 * c, r);
                    tmem_wait_ld_regs16(r);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int col = 16 * c + k;
                        if (col < R_seg) slot[(size_t)col * D + h * 128 + kl] = __uint_as_float(r[k]);
                    }
                }
            }
            tc_fence_before();
        }
        if (bad) set_abort(ms, a.status);
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D, bool BF16, int RGP, int VQ, int KQ>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq, const CUtensorMap& tve,
                       const CUtensorMap& tq2, const AttnLaunch& L, cudaStream_t stream) {
    using Lay = Layout<D, RGP>;
    auto kern = prefix_tc_kernel<D, BF16, RGP, VQ, KQ>;
    static SmemLimitSeen seen;
    cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(kern), Lay::kBytes, seen);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid_ctas(L.plan)), dim3(kThreads), Lay::kBytes, stream, tk, tv, tq, tve, tq2, L);
}

// tve: the per-token exponents of quantised V (VQ != 0); tq2: the low query
// parts of E4M3 K (KQ != 0); unused otherwise
template <int D, bool BF16, int VQ = 0, int KQ = 0>
cudaError_t launch_rgp(int rgp, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                       const CUtensorMap& tve, const CUtensorMap& tq2, const AttnLaunch& L, cudaStream_t stream) {
    static_assert(kRowsMax == 144, "one instantiation per padded row count up to kRowsMax");
    switch (rgp) {
        case 16: return launch_one<D, BF16, 16, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 32: return launch_one<D, BF16, 32, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 48: return launch_one<D, BF16, 48, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 64: return launch_one<D, BF16, 64, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 80: return launch_one<D, BF16, 80, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 96: return launch_one<D, BF16, 96, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 112: return launch_one<D, BF16, 112, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 128: return launch_one<D, BF16, 128, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
        case 144: return launch_one<D, BF16, 144, VQ, KQ>(tk, tv, tq, tve, tq2, L, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace prefix_tc

// tve: the exponent map of quantised V; vq: 0 = 16-bit V, 1 = int8 codes, 2 = int4 codes (head dim 256)
cudaError_t launch_prefix_tc_bf16_256(int rgp, int vq, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const CUtensorMap&, const AttnLaunch&, cudaStream_t);
// E4M3 K (codes map tk, query parts tq / tq2) with V as vq above; bf16, head dim 256
cudaError_t launch_prefix_tc_bf16_256_kq(int rgp, int vq, const CUtensorMap& tk, const CUtensorMap& tv,
                                         const CUtensorMap& tq, const CUtensorMap& tve, const CUtensorMap& tq2,
                                         const AttnLaunch&, cudaStream_t);
cudaError_t launch_prefix_tc_bf16_128(int rgp, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                      const AttnLaunch&, cudaStream_t);
cudaError_t launch_prefix_tc_f16_256(int rgp, int vq, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                     const CUtensorMap&, const AttnLaunch&, cudaStream_t);
cudaError_t launch_prefix_tc_f16_128(int rgp, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                     const AttnLaunch&, cudaStream_t);

}  // namespace lucetree
