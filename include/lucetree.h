/*
 * lucetree.h -- C ABI of the DDTree verify step on one GB300 (sm_103a).
 *
 * One speculative-decoding verify step, as the Lucebox pages describe it:
 * the target checks a whole tree of draft candidates in one forward pass
 * instead of a chain ("Lucebox Hub" (Donggyun's knowledge base), section
 * "Speculative decoding 계층 (DFlash / DDTree / DSpark)"), decoding is greedy at
 * temperature 0 (PyTorch Korea forum post "Lucebox: 추측 디코딩과 전용 커널로 ...",
 * section "Lucebox 설치 및 실행", which also gives the budgets 22 and 40), the
 * KV of rejected tokens is rolled back (the DFlashTarget duties in the
 * "Lucebox Hub" section above), and KV lives in 64-token chunks (forum post,
 * section "Lucebox의 최적화 구성요소"; "Lucebox Hub", section "KVFlash") of a
 * paged pool with a per-sequence block table and D=256 GQA heads ("Lucebox
 * Hub", section "Paged attention + continuous batching").
 *
 * The step is four calls, all asynchronous on the caller's CUDA stream:
 *   lucetree_verify_attn  tree attention: committed prefix + ancestor block
 *   lucetree_argmax       per-node argmax over the vocabulary
 *   lucetree_accept       longest matching root path, greedy
 *   lucetree_commit       copy accepted K/V into the pool, advance lengths
 * plus lucetree_build_anc_mask, which turns a parent array into the ancestor
 * bitmasks verify_attn consumes; lucetree_verify_step runs all of them as one
 * call in two launches.  lucetree_lmhead_argmax replaces
 * the logits + lucetree_argmax pair by the lm_head projection with a fused
 * argmax.  For targets with recurrent (gated delta rule) layers,
 * lucetree_delta_tree advances a layer's state along the tree and
 * lucetree_delta_commit keeps the accepted node's state.  For KV pages kept
 * in host memory, lucetree_stage_pages brings them into the device pool.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers unless a parameter says "host".
 *     The caller owns every buffer; the library allocates no device memory
 *     and keeps no state beyond cached device properties and TMA descriptors
 *     built inside the call.  Calls on different streams do not interfere
 *     as long as their buffers do not overlap.
 *   - Host-detectable errors (null pointers, unsupported sizes, a workspace
 *     that is too small) return an error code before anything is launched.
 *   - Data-dependent errors found by the kernels are OR-ed into the caller's
 *     device status word (uint32_t, LUCETREE_DEV_* flags); kernels never
 *     trap.  A call whose inputs raise a flag still completes; outputs that
 *     depended on the bad input are unspecified.  Clear the word before a
 *     step and read it whenever convenient.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Calls act on the device (and context) current in the calling thread.
 *     One process may drive several GPUs: the kernels that need more than
 *     48 KB of shared memory get that limit raised once per context, and the
 *     split plans follow the current device's SM count.
 */
#ifndef LUCETREE_H
#define LUCETREE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LUCETREE_API __attribute__((visibility("default")))
#else
#define LUCETREE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lucetree_status {
    LUCETREE_OK = 0,
    LUCETREE_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size */
    LUCETREE_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels implement */
    LUCETREE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
    LUCETREE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    LUCETREE_ERR_DEVICE_CHECK = 5, /* reserved: a device status word was non-zero */
    LUCETREE_ERR_TIMEOUT = 6       /* reserved: a bounded device wait gave up */
} lucetree_status;

typedef enum lucetree_dtype {
    LUCETREE_F16 = 0,  /* IEEE binary16 */
    LUCETREE_BF16 = 1  /* bfloat16 */
} lucetree_dtype;

/* Flags kernels OR into the device status word. */
#define LUCETREE_DEV_BAD_PARENT 0x1u /* parent[i] not in [-1, i) */
#define LUCETREE_DEV_BAD_PAGE 0x2u   /* page id outside [0, num_pages) or page index past the table */
#define LUCETREE_DEV_BAD_CTX 0x4u    /* ctx_len outside [0, max_pages_per_seq * 64] */
#define LUCETREE_DEV_BAD_TOKEN 0x8u  /* draft token outside [0, vocab) */
#define LUCETREE_DEV_BAD_NODE 0x10u  /* accepted node id / count out of range, or a mask without self */
#define LUCETREE_DEV_TIMEOUT 0x20u   /* a bounded wait inside a kernel gave up */
#define LUCETREE_DEV_NONFINITE 0x40u /* an attention output is inf or NaN: non-finite inputs, or a bf16 V value
                                        of magnitude >= 65536 (beyond the fp16 range of the on-chip PV product) */

#define LUCETREE_PAGE_SIZE 64 /* tokens per KV page */
#define LUCETREE_MAX_NODES 64 /* tree budget limit (one 64-bit ancestor mask per node) */

/*
 * Arguments of lucetree_verify_attn.  Sizes: B sequences, N tree nodes
 * (1..64), Hq query heads, Hkv KV heads (Hq % Hkv == 0 and Hq / Hkv <= 144;
 * query head h reads KV head h / (Hq / Hkv)), D head dim (128 or 256).
 */
typedef struct lucetree_attn_args {
    int dtype;             /* lucetree_dtype of q, pools and tree K/V */
    int B, N, Hq, Hkv, D;
    int page_size;         /* must be LUCETREE_PAGE_SIZE */
    float scale;           /* softmax scale applied to q.k (1/sqrt(D) in the usual case) */
    const void* q;         /* [B][N][Hq][D], post-RoPE queries of the tree nodes */
    const void* k_pool;    /* [num_pages][Hkv][page_size][D] committed keys */
    const void* v_pool;    /* [num_pages][Hkv][page_size][D] committed values */
    int num_pages;
    const int32_t* page_table; /* [B][max_pages_per_seq]: logical page -> pool page */
    int max_pages_per_seq;
    const int32_t* ctx_len;    /* [B] committed length L_b; positions [0, L_b) are visible */
    const void* k_tree;        /* [B][N][Hkv][D] keys of the tree nodes */
    const void* v_tree;        /* [B][N][Hkv][D] values of the tree nodes */
    const uint64_t* anc_mask;  /* [B][N]: bit j of node i set iff j is i or an ancestor of i */
    float* out;                /* [B][N][Hq][D] fp32 attention output */
    float* lse;                /* [B][N][Hq] natural-log log-sum-exp of the scores, or NULL */
    uint32_t* status;          /* device status word (LUCETREE_DEV_* flags), required */
} lucetree_attn_args;

/*
 * Workspace bytes lucetree_verify_attn needs for these sizes on the CURRENT
 * device (the split plan is sized to its SM count).  The workspace holds
 * per-split partial (O, max, sum) triples; it needs no initialisation and
 * must be 256-byte aligned.  Returns LUCETREE_ERR_UNSUPPORTED for shapes the
 * kernels do not implement.
 */
LUCETREE_API lucetree_status lucetree_verify_attn_workspace(int B, int N, int Hq, int Hkv, int D, size_t* bytes);

/*
 * Tree-verify attention.  For sequence b, node i and query head h:
 *   out[b][i][h] = softmax_j(scale * q.k_j) . v_j
 * over j = every committed position of sequence b (read through the page
 * table) and every tree node j with bit j of anc_mask[b][i] set.  Split-K over
 * the committed prefix on the tensor cores, then one merge launch that adds
 * the tree block and combines the splits by log-sum-exp.
 * Scores and sums are fp32; the P.V product runs on fp16 operands on chip
 * (P rounded to fp16, bf16 V converted exactly while |v| < 65536).
 * Device checks: ctx_len outside [0, max_pages_per_seq*64] -> BAD_CTX (the
 * sequence is treated as empty); page id out of range -> BAD_PAGE (those keys
 * are skipped); a mask without its own bit -> BAD_NODE; an output row that is
 * not finite -> NONFINITE.
 */
LUCETREE_API lucetree_status lucetree_verify_attn(const lucetree_attn_args* args, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* Size of the device array that backs lucetree_verify_attn_noalloc: 32 MiB. */
#define LUCETREE_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * lucetree_verify_attn without a caller-supplied workspace.  The Lucebox
 * pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory: a serving process that has handed all free device
 * memory to its KV page pool up front, or a plugin / foreign-language host
 * that only receives raw device pointers and has no allocator of its own.
 * It computes exactly what lucetree_verify_attn computes (same kernels), and
 * allocates nothing: the split-K partials go to a file-scope device array of
 * 32 MiB (33554432 bytes, LUCETREE_NOALLOC_SCRATCH_BYTES) inside this
 * library, which every GPU that loads the library keeps until the process
 * exits.
 *   - Sizes whose workspace (lucetree_verify_attn_workspace) exceeds 32 MiB
 *     are rejected with LUCETREE_ERR_WORKSPACE before anything is launched;
 *     other errors are those of lucetree_verify_attn.
 *   - Every call looks up the array's device address in the calling thread's
 *     current context, so a device reset or a second context on the device
 *     is followed correctly.  The first call in a context (made with the
 *     target device current) may load the library's device code to do so;
 *     make that first call before any stream capture.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents (the kernels need none of it cleared).  Calls whose
 *     work overlaps on the GPU (different streams, or host threads without
 *     ordering) race on it; serialise them.
 */
LUCETREE_API lucetree_status lucetree_verify_attn_noalloc(const lucetree_attn_args* args, void* stream);

/*
 * anc[b][i] = bit i | anc[b][parent[b][i]] (parent -1 = the root, which holds
 * no bit).  Requires parent[b][i] in [-1, i) (topological order); otherwise
 * BAD_PARENT is raised and anc[b][i] holds bit i only.  parent [B][N],
 * anc [B][N].  N <= 64.
 */
LUCETREE_API lucetree_status lucetree_build_anc_mask(const int32_t* parent, int B, int N, uint64_t* anc, uint32_t* status,
                                        void* stream);

/* Workspace bytes lucetree_argmax needs for `rows` rows of `vocab` entries. */
LUCETREE_API lucetree_status lucetree_argmax_workspace(int rows, int vocab, size_t* bytes);

/*
 * out_idx[r] = the lowest index k with logits[r*row_stride + k] maximal over
 * k in [0, vocab) (ties, including -0.0 vs +0.0, go to the lower index; NaN
 * is outside the contract).  logits fp32, row_stride >= vocab elements.  The
 * workspace (see lucetree_argmax_workspace, 256-byte aligned) needs no
 * initialisation.
 */
LUCETREE_API lucetree_status lucetree_argmax(const float* logits, int rows, int vocab, long long row_stride, int32_t* out_idx,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * Greedy acceptance at temperature 0.  parent, draft [B][N]; argmax
 * [B][N + 1] where row 0 is the root (last committed token) and row j + 1
 * is node j.  Node c matches when draft[c] == argmax row of parent(c).  The
 * accepted path ends at the deepest node whose whole root path matches (the
 * lowest node id among equally deep ones).  Outputs: acc_nodes [B][N] the
 * path root-to-leaf, padded with -1; acc_len [B]; bonus [B] = argmax row of
 * the last accepted node (the root's row when none is accepted).
 * Device checks: BAD_PARENT (the sequence then accepts nothing), BAD_TOKEN
 * (draft outside [0, vocab): never matches).
 */
LUCETREE_API lucetree_status lucetree_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int B, int N,
                                int vocab, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus, uint32_t* status,
                                void* stream);

/* Arguments of lucetree_commit (sizes as in lucetree_attn_args). */
typedef struct lucetree_commit_args {
    int dtype;
    int B, N, Hkv, D;
    int page_size;             /* must be LUCETREE_PAGE_SIZE */
    const void* k_tree;        /* [B][N][Hkv][D] */
    const void* v_tree;        /* [B][N][Hkv][D] */
    const int32_t* acc_nodes;  /* [B][N] from lucetree_accept */
    const int32_t* acc_len;    /* [B] */
    const int32_t* page_table; /* [B][max_pages_per_seq]; must already map positions [L_b, L_b + N) */
    int max_pages_per_seq;
    int num_pages;
    const int32_t* ctx_len_in; /* [B] L_b before the step */
    int32_t* ctx_len_out;      /* [B] L_b + accepted count; may alias ctx_len_in */
    void* k_pool;              /* [num_pages][Hkv][page_size][D], updated in place */
    void* v_pool;
    uint32_t* status;
} lucetree_commit_args;

/*
 * Commit / rollback.  The k-th accepted node's K and V rows (every KV head)
 * are copied to logical position L_b + k: pool page page_table[b][(L_b+k)/64],
 * slot (L_b+k) % 64.  Rejected nodes are never written, which is the
 * rollback.  No other pool byte changes.  ctx_len_out[b] = L_b + count
 * copied.  Device checks: BAD_NODE (count outside [0, N] or node id outside
 * [0, N)), BAD_PAGE, BAD_CTX; copying stops at the first bad entry.
 */
LUCETREE_API lucetree_status lucetree_commit(const lucetree_commit_args* args, void* stream);

/* Arguments of lucetree_verify_step (sizes as in lucetree_attn_args). */
typedef struct lucetree_step_args {
    lucetree_attn_args attn; /* as for lucetree_verify_attn, except: attn.anc_mask is not read (the step
                                derives each node's ancestors from `parent`; NULL is fine), and the pools
                                are also written (the commit) */
    const int32_t* parent;   /* [B][N], parent[b][i] in [-1, i) (-1 = the root) */
    const int32_t* draft;    /* [B][N] draft token of each node */
    const float* logits;     /* [B][N + 1][vocab] fp32; row 0 = the root, row j + 1 = node j */
    int vocab;
    int32_t* argmax;         /* [B][N + 1] out, as lucetree_argmax */
    int32_t* acc_nodes;      /* [B][N] out, as lucetree_accept */
    int32_t* acc_len;        /* [B] out */
    int32_t* bonus;          /* [B] out */
    int32_t* ctx_len_out;    /* [B] out: attn.ctx_len + accepted count; must not alias attn.ctx_len */
} lucetree_step_args;

/*
 * Workspace bytes lucetree_verify_step needs for these sizes on the CURRENT
 * device.  Its first bytes past the attention partials hold counters that
 * must be ZERO before the first call on a workspace (allocate it zeroed);
 * every call leaves them zero again.  256-byte aligned.
 */
LUCETREE_API lucetree_status lucetree_verify_step_workspace(int B, int N, int Hq, int Hkv, int D, int vocab,
                                                            size_t* bytes);

/*
 * The whole verify step in one call: what lucetree_build_anc_mask,
 * lucetree_verify_attn, lucetree_argmax, lucetree_accept and lucetree_commit
 * compute in sequence, with the same results, in two launches.  The first is
 * the attention's split-K prefix kernel; the second runs the argmax chunks
 * (while the prefix kernel's last CTAs still stream K/V), the acceptance and
 * commit of each sequence (by the CTA that completes its last argmax row,
 * after the prefix kernel has completed) and the attention merge, with each
 * node's ancestors walked from `parent`.  The pages describe these steps
 * (greedy verification of the whole tree, then KV rollback of the rejected
 * nodes: "Lucebox Hub", section "Speculative decoding 계층"; forum post,
 * section "Lucebox 설치 및 실행"); fusing them is this library's.
 * Errors: those of the five calls; INVALID_ARG also when ctx_len_out aliases
 * attn.ctx_len; UNSUPPORTED when B * (N + 1) > 65535.  Device checks as the
 * five calls (BAD_PARENT is raised once per bad node).
 */
LUCETREE_API lucetree_status lucetree_verify_step(const lucetree_step_args* args, void* workspace,
                                                  size_t workspace_bytes, void* stream);

/* K storage formats (lucetree_verify_attn_kq, lucetree_commit_kq). */
#define LUCETREE_K_SAME 0 /* K in the args' 16-bit dtype */
#define LUCETREE_K_E4M3 1 /* FP8 E4M3 codes [num_pages][Hkv][64][D], value = e4m3(code) * 2^(e - 127) */

/* V storage formats of lucetree_verify_attn_vq (K stays in the args' dtype). */
#define LUCETREE_V_SAME 0 /* V in the args' 16-bit dtype (lucetree_verify_attn) */
#define LUCETREE_V_INT8 1 /* int8 codes [num_pages][Hkv][64][D], value = code * 2^(e - 127) */
#define LUCETREE_V_INT4 2 /* int4 codes [num_pages][Hkv][64][D / 2], two per byte, low nibble = even dim */

/*
 * lucetree_verify_attn with V held quantised: asymmetric K/V storage, K in
 * the 16-bit dtype and V as small integer codes with one power-of-two scale
 * per token and head.  The pages list KV quantisation, TQ3_0 and asymmetric
 * K/V quantisation among the project's components ("Lucebox Hub", section
 * "Speculative decoding 계층"; pytorch.kr Lucebox introduction, section
 * "Lucebox의 최적화 구성요소") without defining a format.  This one is the
 * library's own:
 *   - a->v_pool holds the codes (format v_format): int8 in [-127, 127], or
 *     two's-complement int4 in [-7, 7];
 *   - v_exp [num_pages][Hkv][64] holds one exponent byte e per token and KV
 *     head (16-byte aligned); the value is code * 2^(e - 127), e = 0 means 0.
 * Every such value with e in [103, 135] is exact in fp16, which is the
 * on-chip type of the PV product; elsewhere precision or range is lost.  The
 * tree's own V (a->v_tree) stays in the 16-bit dtype.  Head dim 256 only.
 * Errors as lucetree_verify_attn, plus UNSUPPORTED (v_format, D != 256) and
 * INVALID_ARG (v_exp null or misaligned).
 */
LUCETREE_API lucetree_status lucetree_verify_attn_vq(const lucetree_attn_args* args, int v_format,
                                                     const uint8_t* v_exp, void* workspace, size_t workspace_bytes,
                                                     void* stream);

/*
 * Workspace bytes lucetree_verify_attn_kq needs on the CURRENT device: the
 * attention partials plus the two E4M3 parts of the scaled queries (B*N*Hq*D
 * bytes each) and one float per key segment.  Needs no initialisation;
 * 256-byte aligned.  UNSUPPORTED for shapes without a kernel (D != 256).
 */
LUCETREE_API lucetree_status lucetree_verify_attn_kq_workspace(int B, int N, int Hq, int Hkv, int D,
                                                               size_t* bytes);

/*
 * lucetree_verify_attn with K held as FP8 E4M3 codes: asymmetric K/V storage
 * on the K side (the pages list KV quantisation, TQ3_0 and asymmetric K/V
 * quantisation among the project's components without defining a format:
 * "Lucebox Hub", section "Speculative decoding 계층"; forum post, section
 * "Lucebox의 최적화 구성요소"; this format is the library's own):
 *   - a->k_pool holds the codes [num_pages][Hkv][64][D] (uint8);
 *   - k_exp [num_pages][Hkv][64] holds one exponent byte e per token and KV
 *     head (16-byte aligned); the value is e4m3(code) * 2^(e - 127), e = 0
 *     reads as zero, e = 255 and the NaN codes (0x7F, 0xFF) are outside the
 *     contract;
 *   - V as in lucetree_verify_attn (v_format LUCETREE_V_SAME) or as the codes
 *     of lucetree_verify_attn_vq (LUCETREE_V_INT8 / LUCETREE_V_INT4 with v_exp).
 * QK runs on the FP8 tensor cores with the queries of each (sequence, KV
 * head) scaled by one power of two and split into two E4M3 parts, which
 * reproduce exactly every bf16 query element whose scaled magnitude is at
 * least 1/4 (the largest lies in (224, 448]; smaller elements are off by at
 * most 2^-10 of the scaled unit);
 * the tree's own K/V (k_tree, v_tree) stay bf16.  bf16 queries, D = 256.
 * Errors as lucetree_verify_attn, plus UNSUPPORTED (dtype, D, v_format) and
 * INVALID_ARG (k_exp / v_exp null or misaligned).
 */
LUCETREE_API lucetree_status lucetree_verify_attn_kq(const lucetree_attn_args* args, const uint8_t* k_exp,
                                                     int v_format, const uint8_t* v_exp, void* workspace,
                                                     size_t workspace_bytes, void* stream);

/*
 * lucetree_commit into a K pool held as E4M3 codes (args->k_pool: codes
 * [num_pages][Hkv][64][D], k_exp [num_pages][Hkv][64]) with V in bf16: the
 * k-th accepted node's K row of each KV head is stored at position L_b + k as
 * its codes and exponent: e = 127 - p with p the largest integer such that
 * max|k| * 2^p <= 448, code_d = e4m3(k_d * 2^p) rounded to nearest, ties to
 * the even code.  A row of zeros, or one whose largest magnitude is below
 * 2^-118 (e would leave [1, 254]), is stored as zero (e = 0).  V rows, the
 * length update, the rollback and the device checks are those of
 * lucetree_commit.  bf16, D = 256.
 */
LUCETREE_API lucetree_status lucetree_commit_kq(const lucetree_commit_args* args, uint8_t* k_exp, void* stream);

/* Arguments of lucetree_lmhead_argmax. */
typedef struct lucetree_lmhead_args {
    int dtype;             /* LUCETREE_F16 / LUCETREE_BF16, both operands */
    int rows;              /* R = B * (N + 1) verify rows (root + nodes), 1..256 */
    int d_model;           /* hidden size, a positive multiple of 64 */
    int vocab;             /* >= 1 */
    const void* hidden;    /* [rows][d_model], 16-byte aligned */
    const void* weight;    /* [vocab][d_model] lm_head weight, 16-byte aligned */
    int32_t* out_idx;      /* [rows] */
    float* out_logit;      /* [rows] the maximal logit (fp32 accumulation), or NULL */
    uint32_t* status;
} lucetree_lmhead_args;

/* Workspace bytes lucetree_lmhead_argmax needs for `rows` rows (host output). */
LUCETREE_API lucetree_status lucetree_lmhead_argmax_workspace(int rows, size_t* bytes);

/*
 * The target's lm_head projection fused with the argmax: out_idx[r] = the
 * lowest v with sum_d hidden[r][d] * weight[v][d] maximal, without writing
 * the logits.  The pages list projecting hidden states through the target's
 * lm_head as one DFlashTarget duty ("Lucebox Hub", section "Speculative
 * decoding 계층"); the fused form, its layout and its sizes are this
 * library's.  Accumulation is fp32 on the tensor cores, so rows whose two
 * best logits lie within that rounding may pick either (a NaN logit is
 * outside the contract).  The workspace (256-byte aligned, see
 * lucetree_lmhead_argmax_workspace) is cleared by the call itself.  Host
 * errors: INVALID_ARG (null or misaligned pointers, sizes out of range),
 * UNSUPPORTED (rows > 256, d_model not a multiple of 64), WORKSPACE.
 * Device check: TIMEOUT.
 */
LUCETREE_API lucetree_status lucetree_lmhead_argmax(const lucetree_lmhead_args* args, void* workspace,
                                                    size_t workspace_bytes, void* stream);

/* Arguments of lucetree_delta_tree and lucetree_delta_commit. */
typedef struct lucetree_delta_args {
    int dtype;               /* LUCETREE_F16 / LUCETREE_BF16: q, k, v */
    int B, N;                /* sequences; tree nodes 1..64 */
    int Hk, Hv;              /* query/key heads, value heads (Hv % Hk == 0) */
    int dk, dv;              /* head dims: dk = 128, dv a positive multiple of 8 */
    const void* q;           /* [B][N][Hk][dk]; tree pass only */
    const void* k;           /* [B][N][Hk][dk] */
    const void* v;           /* [B][N][Hv][dv] */
    const float* alpha;      /* [B][N][Hv] decay gate */
    const float* beta;       /* [B][N][Hv] write strength */
    const int32_t* parent;   /* [B][N], parent[i] in [-1, i); tree pass only */
    float* state;            /* [B][Hv][dk][dv]: read by the tree pass, updated by the commit */
    float* out;              /* [B][N][Hv][dv]; tree pass only */
    const int32_t* acc_nodes; /* [B][N] accepted path, root first (lucetree_accept); commit only */
    const int32_t* acc_len;   /* [B]; commit only */
    uint32_t* status;        /* device status word, required */
} lucetree_delta_args;

/*
 * One gated-delta-rule (DeltaNet-style) layer over the draft tree.  The pages
 * name a tree-aware DeltaNet rollback kernel for targets that mix DeltaNet
 * and attention layers ("Lucebox Hub", section "Speculative decoding 계층
 * (DFlash / DDTree / DSpark)") without a formula.  This library reads it as
 * follows.  For value head h (query/key head h / (Hv / Hk)), with the
 * committed state as the root's state:
 *     S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T
 *     out_i = S_i^T q_i        (fp32; the state is read, never written)
 * Layouts are row-major; q, k, v 8-byte and state 16-byte aligned.  Host
 * errors: INVALID_ARG, UNSUPPORTED (dk != 128, dv % 8, N > 64).  Device
 * check: BAD_PARENT (that node is then treated as a root child).
 */
LUCETREE_API lucetree_status lucetree_delta_tree(const lucetree_delta_args* args, void* stream);

/*
 * The rollback: state[b] <- the recurrence above run from state[b] over
 * acc_nodes[b][0 .. acc_len[b]) in order, i.e. the accepted node's state.
 * Rejected nodes never touch it; acc_len[b] = 0 leaves it bit for bit.
 * Device check: BAD_NODE (count outside [0, N] or node outside [0, N): that
 * sequence's state is left unchanged).
 */
LUCETREE_API lucetree_status lucetree_delta_commit(const lucetree_delta_args* args, void* stream);

/* Arguments of lucetree_stage_pages. */
typedef struct lucetree_stage_args {
    int Hkv, D;               /* pool geometry: one page of one tensor is [Hkv][64][D] 16-bit values */
    int n;                    /* pages to stage (0: nothing to do) */
    const void* host_k;       /* host-resident pools [host_pages][Hkv][64][D]: page-locked HOST memory */
    const void* host_v;
    int host_pages;
    const int32_t* src;       /* [n] host page ids (device array) */
    const int32_t* dst;       /* [n] device pool page ids to fill (device array), distinct */
    const int32_t* table_idx; /* [n] flat page-table positions (b * max_pages + page) to set to dst, or NULL */
    int32_t* page_table;      /* [table_len] (device), required with table_idx */
    int table_len;
    void* k_pool;             /* device pools [num_pages][Hkv][64][D] */
    void* v_pool;
    int num_pages;
    uint32_t* status;
} lucetree_stage_args;

/*
 * Host-resident cold pages: copy host pages src[i] of both pools into device
 * pool pages dst[i] and, with table_idx, set page_table[table_idx[i]] =
 * dst[i], so that lucetree_verify_attn reads them like any resident page.
 * The pages keep cold 64-token KV chunks in host memory ("Lucebox Hub",
 * section "KVFlash"); the choice of pages and the free-page bookkeeping are
 * the caller's.  The kernel reads the host pools directly (zero copy over
 * the CPU-GPU link); byte-exact.  Host errors: INVALID_ARG (null or
 * misaligned pointers, host pools that are not page-locked host memory,
 * sizes).  Device check: BAD_PAGE (an id or table position out of range:
 * that page is skipped).
 */
LUCETREE_API lucetree_status lucetree_stage_pages(const lucetree_stage_args* args, void* stream);

/*
 * Self-test of the failure path shared by every kernel wait: one block waits
 * on a barrier that nothing arrives on, gives up after ~limit_cycles SM
 * cycles (1 .. 4e9; the step kernels use 4e9, about two seconds), sets
 * LUCETREE_DEV_TIMEOUT in *status and returns.  waited_cycles (device
 * int64, or NULL) receives the cycles the wait took.  Host errors:
 * INVALID_ARG (null status, limit out of range), CUDA.
 */
LUCETREE_API lucetree_status lucetree_selftest_wait_timeout(uint32_t* status, long long limit_cycles,
                                                            long long* waited_cycles, void* stream);

/* Human-readable name of a status code (static storage). */
LUCETREE_API const char* lucetree_status_string(lucetree_status status);

/* ABI version of this header: 1. */
LUCETREE_API int lucetree_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LUCETREE_H */
