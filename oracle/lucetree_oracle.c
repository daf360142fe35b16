/*
 * lucetree_oracle.c -- plain, slow, fp64 CPU reference for the DDTree verify
 * step.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library never does.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes follows the Lucebox pages' statement of DDTree
 * verification: the target checks a tree of draft candidates in one forward
 * pass ("Lucebox Hub", section "Speculative decoding layer (DFlash / DDTree /
 * DSpark)"), greedy acceptance at temperature 0 (pytorch.kr Lucebox
 * introduction, section "Installation and running"), and rejected tokens'
 * K/V are rolled back ("Lucebox Hub", same section, the DFlashTarget duties).
 * The pages give no formulas; where they are silent the plainest reading is
 * taken and listed in the design notes:
 *   - softmax scale is a parameter (1/sqrt(D) in every workload);
 *   - query head h reads KV head h / (Hq / Hkv);
 *   - node i attends every committed key plus tree node j iff j is i or an
 *     ancestor of i (found by walking parent[] up to -1);
 *   - argmax ties go to the lowest index (a strict ">" linear scan);
 *   - acceptance keeps the deepest node whose whole root path matches, the
 *     lowest node index among equally deep ones;
 *   - commit writes accepted node k (root-to-leaf order) at logical position
 *     L_b + k through the page table and adds the accepted count to L_b.
 *
 * Parity pins (tests/test_oracle_pins.py): hand-worked 3-node examples,
 * closed forms (equal keys -> mean of visible V), a one-node tree against an
 * independent textbook decode routine, a chain tree against causal attention,
 * brute-force enumeration of root paths for acceptance, numpy's first-index
 * argmax, and byte-level invariants of the commit copy.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---- exact upcast of the 16-bit storage formats (IEEE 754 binary16, and
 *      bfloat16 = the top half of binary32) ---------------------------------- */

static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);
    return sign ? -v : v;
}

static double bfloat_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 7) & 0xff, m = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x80), e - 134);
    return sign ? -v : v;
}

static double g_table[2][65536];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;
static void fill_tables(void) {
    for (int i = 0; i < 65536; ++i) {
        g_table[ORACLE_F16][i] = half_to_double((uint16_t)i);
        g_table[ORACLE_BF16][i] = bfloat_to_double((uint16_t)i);
    }
}

double oracle_upcast(int dtype, uint16_t bits) {
    pthread_once(&g_once, fill_tables);
    return g_table[dtype ? ORACLE_BF16 : ORACLE_F16][bits];
}

/* ---- tree structure ------------------------------------------------------- */

/* 1 iff node j is node i or one of its ancestors: walk parent[] from i to -1. */
static int is_ancestor_or_self(const int32_t* parent, int N, int j, int i) {
    int cur = i, steps = 0;
    while (cur >= 0 && steps <= N) {
        if (cur == j) return 1;
        cur = parent[cur];
        ++steps;
    }
    return 0;
}

/* anc[i * N + j] = 1 iff j is i or an ancestor of i. */
void oracle_ancestor_matrix(const int32_t* parent, int N, uint8_t* anc) {
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) anc[(size_t)i * N + j] = (uint8_t)is_ancestor_or_self(parent, N, j, i);
}

/* ---- tree-verify attention -------------------------------------------------- */

typedef struct {
    int dtype, B, N, Hq, Hkv, D, page_size;
    double scale;
    const uint16_t *q, *k_pool, *v_pool, *k_tree, *v_tree;
    int num_pages;
    const int32_t* page_table;
    int max_pages;
    const int32_t *ctx_len, *parent;
    const int32_t* rows; /* flat row ids ((b*N + i)*Hq + h), or NULL = all */
    long num_rows;
    double *out, *lse;
    int num_threads, tid;
    int error;
} attn_job;

/* One output row: explicit visibility mask over the L + N positions, then
 * softmax(q . k * scale) over the visible ones and the weighted sum of V. */
static int attn_row(const attn_job* a, long row, double* out, double* lse_out,
                    unsigned char* vis, double* s) {
    const double* T = g_table[a->dtype ? ORACLE_BF16 : ORACLE_F16];
    const int N = a->N, Hq = a->Hq, Hkv = a->Hkv, D = a->D, P = a->page_size;
    const int h = (int)(row % Hq);
    const int i = (int)((row / Hq) % N);
    const int b = (int)(row / ((long)Hq * N));
    const int g = h / (Hq / Hkv);
    const int L = a->ctx_len[b];
    const int32_t* par = a->parent + (size_t)b * N;
    const uint16_t* qv = a->q + (((size_t)b * N + i) * Hq + h) * D;

    /* explicit mask: every committed position, and tree slot j iff j is i or an ancestor */
    for (int j = 0; j < L; ++j) vis[j] = 1;
    for (int j = 0; j < N; ++j) vis[L + j] = (unsigned char)is_ancestor_or_self(par, N, j, i);

    double qd[1024];
    for (int d = 0; d < D; ++d) qd[d] = T[qv[d]];

    double mx = -INFINITY;
    for (int j = 0; j < L + N; ++j) {
        if (!vis[j]) continue;
        const uint16_t* kv;
        if (j < L) {
            int page = a->page_table[(size_t)b * a->max_pages + j / P];
            if (page < 0 || page >= a->num_pages) return -1;
            kv = a->k_pool + (((size_t)page * Hkv + g) * P + (j % P)) * D;
        } else {
            kv = a->k_tree + (((size_t)b * N + (j - L)) * Hkv + g) * D;
        }
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * T[kv[d]];
        s[j] = dot * a->scale;
        if (s[j] > mx) mx = s[j];
    }
    double sum = 0.0;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int j = 0; j < L + N; ++j) {
        if (!vis[j]) continue;
        const uint16_t* vv;
        if (j < L) {
            int page = a->page_table[(size_t)b * a->max_pages + j / P];
            vv = a->v_pool + (((size_t)page * Hkv + g) * P + (j % P)) * D;
        } else {
            vv = a->v_tree + (((size_t)b * N + (j - L)) * Hkv + g) * D;
        }
        double p = exp(s[j] - mx);
        sum += p;
        for (int d = 0; d < D; ++d) out[d] += p * T[vv[d]];
    }
    for (int d = 0; d < D; ++d) out[d] /= sum;
    if (lse_out) *lse_out = mx + log(sum);
    return 0;
}

static void* attn_worker(void* arg) {
    attn_job* a = (attn_job*)arg;
    int maxL = 0;
    for (int b = 0; b < a->B; ++b)
        if (a->ctx_len[b] > maxL) maxL = a->ctx_len[b];
    unsigned char* vis = (unsigned char*)malloc((size_t)maxL + a->N + 1);
    double* s = (double*)malloc(sizeof(double) * ((size_t)maxL + a->N + 1));
    if (!vis || !s) { a->error = -2; free(vis); free(s); return NULL; }
    for (long r = a->tid; r < a->num_rows; r += a->num_threads) {
        long row = a->rows ? a->rows[r] : r;
        if (attn_row(a, row, a->out + (size_t)r * a->D, a->lse ? a->lse + r : NULL, vis, s) != 0) {
            a->error = -1;
            break;
        }
    }
    free(vis);
    free(s);
    return NULL;
}

/*
 * q [B][N][Hq][D]; k_pool, v_pool [num_pages][Hkv][page_size][D];
 * page_table [B][max_pages]; ctx_len [B]; k_tree, v_tree [B][N][Hkv][D];
 * parent [B][N] (-1 = root).  rows: flat ids of the rows to compute (NULL =
 * all B*N*Hq in order).  out [num_rows][D] fp64, lse [num_rows] (natural log,
 * may be NULL).  Returns 0, or -1 on an out-of-range page id, -2 on OOM,
 * -3 on bad sizes.
 */
int oracle_verify_attn(int dtype, int B, int N, int Hq, int Hkv, int D, int page_size, double scale,
                       const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool, int num_pages,
                       const int32_t* page_table, int max_pages, const int32_t* ctx_len,
                       const uint16_t* k_tree, const uint16_t* v_tree, const int32_t* parent,
                       const int32_t* rows, long num_rows, double* out, double* lse, int num_threads) {
    pthread_once(&g_once, fill_tables);
    if (D <= 0 || D > 1024 || Hkv <= 0 || Hq % Hkv != 0 || N <= 0 || page_size <= 0) return -3;
    if (!rows) num_rows = (long)B * N * Hq;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 512) num_threads = 512;
    attn_job* jobs = (attn_job*)calloc((size_t)num_threads, sizeof(attn_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int t = 0; t < num_threads; ++t) {
        attn_job* a = &jobs[t];
        a->dtype = dtype; a->B = B; a->N = N; a->Hq = Hq; a->Hkv = Hkv; a->D = D;
        a->page_size = page_size; a->scale = scale; a->q = q; a->k_pool = k_pool; a->v_pool = v_pool;
        a->k_tree = k_tree; a->v_tree = v_tree; a->num_pages = num_pages; a->page_table = page_table;
        a->max_pages = max_pages; a->ctx_len = ctx_len; a->parent = parent; a->rows = rows;
        a->num_rows = num_rows; a->out = out; a->lse = lse; a->num_threads = num_threads; a->tid = t;
    }
    for (int t = 1; t < num_threads; ++t) pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    attn_worker(&jobs[0]);
    for (int t = 1; t < num_threads; ++t) pthread_join(th[t], NULL);
    int err = 0;
    for (int t = 0; t < num_threads; ++t)
        if (jobs[t].error) err = jobs[t].error;
    free(jobs);
    free(th);
    return err;
}

/* ---- argmax over the vocabulary ---------------------------------------------- */

/* Linear scan per row; a later element wins only if strictly greater, so ties
 * (including -0.0 against +0.0) keep the lowest index. */
void oracle_argmax(const float* logits, long rows, long vocab, long row_stride, int32_t* out) {
    for (long r = 0; r < rows; ++r) {
        const float* x = logits + r * row_stride;
        float best = x[0];
        long idx = 0;
        for (long k = 1; k < vocab; ++k) {
            if (x[k] > best) {
                best = x[k];
                idx = k;
            }
        }
        out[r] = (int32_t)idx;
    }
}

/* ---- greedy acceptance ---------------------------------------------------------- */

/*
 * parent, draft [B][N]; argmax [B][N + 1] (row 0 = root, row j + 1 = node j).
 * Node c "matches" when draft[c] equals the argmax of its parent's row.  A node
 * is acceptable when every node on its root path matches.  The accepted path
 * ends at the deepest acceptable node (lowest index among equals); acc_nodes
 * lists it root-to-leaf, acc_len is its depth, bonus is the argmax of its row
 * (the root's when nothing is accepted).  Returns 0, or -1 on a parent that is
 * not an earlier node or -1.
 */
int oracle_accept(int B, int N, const int32_t* parent, const int32_t* draft, const int32_t* argmax,
                  int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus) {
    for (int b = 0; b < B; ++b) {
        const int32_t* par = parent + (size_t)b * N;
        const int32_t* dr = draft + (size_t)b * N;
        const int32_t* am = argmax + (size_t)b * (N + 1);
        for (int i = 0; i < N; ++i)
            if (par[i] < -1 || par[i] >= i) return -1;
        int best = -1, best_depth = 0;
        for (int i = 0; i < N; ++i) {
            int ok = 1, depth = 0;
            for (int c = i; c >= 0; c = par[c]) {
                ++depth;
                if (dr[c] != am[par[c] + 1]) { ok = 0; break; }
            }
            if (ok && depth > best_depth) {
                best = i;
                best_depth = depth;
            }
        }
        int32_t* out = acc_nodes + (size_t)b * N;
        for (int k = 0; k < N; ++k) out[k] = -1;
        int k = best_depth;
        for (int c = best; c >= 0; c = par[c]) out[--k] = c;
        acc_len[b] = best_depth;
        bonus[b] = am[best + 1];
    }
    return 0;
}

/* ---- commit / rollback ------------------------------------------------------------- */

/*
 * Copy tree K/V rows of the accepted nodes into the pool: the k-th accepted
 * node goes to logical position L_b + k, i.e. page page_table[b][(L_b+k)/P],
 * slot (L_b+k) % P, for every KV head.  Nothing else in the pools changes;
 * ctx_len[b] grows by acc_len[b].  Pools and ctx_len are updated in place.
 * Returns 0, or -1 on an out-of-range page.
 */
int oracle_commit(int B, int N, int Hkv, int D, int page_size, const uint16_t* k_tree,
                  const uint16_t* v_tree, const int32_t* acc_nodes, const int32_t* acc_len,
                  const int32_t* page_table, int max_pages, int num_pages, int32_t* ctx_len,
                  uint16_t* k_pool, uint16_t* v_pool) {
    for (int b = 0; b < B; ++b) {
        int L = ctx_len[b];
        for (int k = 0; k < acc_len[b]; ++k) {
            int node = acc_nodes[(size_t)b * N + k];
            long pos = (long)L + k;
            if (pos / page_size >= max_pages) return -1;
            int page = page_table[(size_t)b * max_pages + pos / page_size];
            if (page < 0 || page >= num_pages) return -1;
            int slot = (int)(pos % page_size);
            for (int g = 0; g < Hkv; ++g) {
                size_t dst = (((size_t)page * Hkv + g) * page_size + slot) * D;
                size_t src = (((size_t)b * N + node) * Hkv + g) * D;
                memcpy(k_pool + dst, k_tree + src, sizeof(uint16_t) * D);
                memcpy(v_pool + dst, v_tree + src, sizeof(uint16_t) * D);
            }
        }
        ctx_len[b] = L + acc_len[b];
    }
    return 0;
}

/* ---- lm_head projection fused with the argmax ---------------------------------
 *
 * The target projects hidden states through its lm_head ("Lucebox Hub", section
 * "Speculative decoding layer", the third DFlashTarget duty); the verify step
 * needs only the argmax of each row's logits.  Definition, on the exactly
 * upcast 16-bit inputs:
 *     logit[r][v] = sum_d hidden[r][d] * weight[v][d]      (fp64)
 *     out[r]      = the lowest v with the largest logit[r][v]
 * top1[r] / top2[r] receive the largest and second-largest logit of row r (the
 * second over the other vocabulary entries), so a caller can tell a clear winner
 * from a near tie that another summation order could decide differently.
 * The vocabulary is split over num_threads threads; each keeps, per row, its
 * slice's best (value, lowest index) and two largest values, merged in slice
 * order.  Returns 0, or -1 on bad sizes / allocation failure.
 */
typedef struct {
    int dtype;
    long rows, d_model, v0, v1;
    const uint16_t* hidden;
    const uint16_t* weight;
    const double* hid;   /* upcast hidden [rows][d_model] */
    double* best;        /* [rows] */
    long* idx;           /* [rows] */
    double* second;      /* [rows] */
} lm_job;

static void* lm_worker(void* arg) {
    lm_job* j = (lm_job*)arg;
    double* w = (double*)malloc(sizeof(double) * (size_t)j->d_model);
    if (!w) return (void*)1;
    for (long r = 0; r < j->rows; ++r) {
        j->best[r] = -INFINITY;
        j->second[r] = -INFINITY;
        j->idx[r] = -1;
    }
    for (long v = j->v0; v < j->v1; ++v) {
        const uint16_t* wr = j->weight + (size_t)v * (size_t)j->d_model;
        for (long d = 0; d < j->d_model; ++d) w[d] = oracle_upcast(j->dtype, wr[d]);
        for (long r = 0; r < j->rows; ++r) {
            const double* h = j->hid + (size_t)r * (size_t)j->d_model;
            double s = 0.0;
            for (long d = 0; d < j->d_model; ++d) s += h[d] * w[d];
            if (s > j->best[r]) {
                j->second[r] = j->best[r];
                j->best[r] = s;
                j->idx[r] = v;
            } else if (s > j->second[r]) {
                j->second[r] = s;
            }
        }
    }
    free(w);
    return NULL;
}

int oracle_lmhead_argmax(int dtype, long rows, long d_model, long vocab, const uint16_t* hidden,
                         const uint16_t* weight, int32_t* out, double* top1, double* top2, int num_threads) {
    if (rows <= 0 || d_model <= 0 || vocab <= 0) return -1;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > vocab) num_threads = (int)vocab;
    double* hid = (double*)malloc(sizeof(double) * (size_t)rows * (size_t)d_model);
    lm_job* jobs = (lm_job*)calloc((size_t)num_threads, sizeof(lm_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    double* best = (double*)malloc(sizeof(double) * (size_t)rows * (size_t)num_threads);
    double* second = (double*)malloc(sizeof(double) * (size_t)rows * (size_t)num_threads);
    long* idx = (long*)malloc(sizeof(long) * (size_t)rows * (size_t)num_threads);
    int err = (!hid || !jobs || !th || !best || !second || !idx) ? -1 : 0;
    if (!err) {
        for (long i = 0; i < rows * d_model; ++i) hid[i] = oracle_upcast(dtype, hidden[i]);
        for (int t = 0; t < num_threads; ++t) {
            lm_job* j = &jobs[t];
            j->dtype = dtype;
            j->rows = rows;
            j->d_model = d_model;
            j->v0 = vocab * t / num_threads;
            j->v1 = vocab * (t + 1) / num_threads;
            j->hidden = hidden;
            j->weight = weight;
            j->hid = hid;
            j->best = best + (size_t)t * (size_t)rows;
            j->idx = idx + (size_t)t * (size_t)rows;
            j->second = second + (size_t)t * (size_t)rows;
            if (pthread_create(&th[t], NULL, lm_worker, j) != 0) {
                err = -1;
                num_threads = t;
                break;
            }
        }
        for (int t = 0; t < num_threads; ++t) {
            void* rv = NULL;
            pthread_join(th[t], &rv);
            if (rv) err = -1;
        }
    }
    if (!err) {
        /* merge the slices in vocabulary order: a later slice wins only if strictly greater */
        for (long r = 0; r < rows; ++r) {
            double b = -INFINITY, s2 = -INFINITY;
            long bi = -1;
            for (int t = 0; t < num_threads; ++t) {
                const double tb = best[(size_t)t * (size_t)rows + r];
                const double ts = second[(size_t)t * (size_t)rows + r];
                const long ti = idx[(size_t)t * (size_t)rows + r];
                if (ti < 0) continue;
                if (tb > b) {
                    s2 = b > ts ? b : ts;
                    b = tb;
                    bi = ti;
                } else {
                    const double c = tb > ts ? tb : ts;
                    if (c > s2) s2 = c;
                }
            }
            out[r] = (int32_t)bi;
            if (top1) top1[r] = b;
            if (top2) top2[r] = s2;
        }
    }
    free(hid);
    free(jobs);
    free(th);
    free(best);
    free(second);
    free(idx);
    return err;
}

/*
 * Tree-aware recurrent-state step (gated delta rule).  The pages name a
 * tree-aware SSM (DeltaNet) rollback kernel among the DFlash components
 * ("Lucebox Hub", section "Speculative decoding layer (DFlash / DDTree /
 * DSpark)") for targets that mix DeltaNet and attention layers, but give no
 * formula.  Reading taken: the gated delta rule with one state S [dk][dv] per
 * value head,
 *     S_i = alpha_i (I - beta_i k_i k_i^T) S_parent(i) + beta_i k_i v_i^T,
 *     o_i = S_i^T q_i,
 * where the root's S (parent -1) is the committed state and value head h
 * reads query/key head h / (Hv / Hk).  Each node's output follows from the
 * recurrence run from the committed state along that node's root path (found
 * by walking parent[]), one node at a time; the commit runs it along the
 * accepted path and stores the result, so rejected nodes leave no trace.
 */
static int delta_path(const int32_t* parent, int N, int i, int* path) {
    int n = 0;
    for (int j = i; j != -1; j = parent[j]) {
        if (j < -1 || j >= N || n >= N) return -1;
        if (j != i && j >= path[n - 1]) return -1; /* parents come before children */
        path[n++] = j;
    }
    /* root first */
    for (int a = 0, b = n - 1; a < b; ++a, --b) {
        const int t = path[a];
        path[a] = path[b];
        path[b] = t;
    }
    return n;
}

/* S <- alpha (I - beta k k^T) S + beta k v^T, S [dk][dv] row-major */
static void delta_update(int dk, int dv, double* S, const double* k, const double* v, double alpha, double beta,
                         double* u) {
    for (int j = 0; j < dv; ++j) {
        double s = 0.0;
        for (int r = 0; r < dk; ++r) s += k[r] * S[(size_t)r * dv + j];
        u[j] = s; /* (k^T S)_j */
    }
    for (int r = 0; r < dk; ++r)
        for (int j = 0; j < dv; ++j) {
            double* x = &S[(size_t)r * dv + j];
            *x = alpha * (*x - beta * k[r] * u[j]) + beta * k[r] * v[j];
        }
}

static void delta_load(int dtype, const uint16_t* src, int n, double* dst) {
    for (int x = 0; x < n; ++x) dst[x] = oracle_upcast(dtype, src[x]);
}

/*
 * q, k [B][N][Hk][dk], v [B][N][Hv][dv] (16-bit bits of dtype), alpha, beta
 * [B][N][Hv], parent [B][N], state [B][Hv][dk][dv] (fp32) -> out [B][N][Hv][dv].
 * Returns 0, or -1 on a bad parent array / sizes / allocation failure.
 */
int oracle_delta_tree(int dtype, int B, int N, int Hk, int Hv, int dk, int dv, const uint16_t* q,
                      const uint16_t* k, const uint16_t* v, const float* alpha, const float* beta,
                      const int32_t* parent, const float* state, double* out) {
    if (B < 1 || N < 1 || Hk < 1 || Hv < 1 || Hv % Hk != 0 || dk < 1 || dv < 1) return -1;
    const int G = Hv / Hk;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dk);
    double* qq = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    int* path = (int*)malloc(sizeof(int) * (size_t)N);
    int err = (!S || !u || !kk || !qq || !vv || !path) ? -1 : 0;
    for (int b = 0; b < B && !err; ++b)
        for (int h = 0; h < Hv && !err; ++h) {
            const int hk = h / G;
            for (int i = 0; i < N && !err; ++i) {
                const int n = delta_path(parent + (size_t)b * N, N, i, path);
                if (n < 0) {
                    err = -1;
                    break;
                }
                const float* s0 = state + ((size_t)b * Hv + h) * (size_t)dk * dv;
                for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] = s0[x];
                for (int t = 0; t < n; ++t) {
                    const size_t node = (size_t)b * N + path[t];
                    delta_load(dtype, k + (node * Hk + hk) * dk, dk, kk);
                    delta_load(dtype, v + (node * Hv + h) * dv, dv, vv);
                    delta_update(dk, dv, S, kk, vv, alpha[node * Hv + h], beta[node * Hv + h], u);
                }
                const size_t node = (size_t)b * N + i;
                delta_load(dtype, q + (node * Hk + hk) * dk, dk, qq);
                double* o = out + (node * Hv + h) * dv;
                for (int j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (int r = 0; r < dk; ++r) s += qq[r] * S[(size_t)r * dv + j];
                    o[j] = s;
                }
            }
        }
    free(S);
    free(u);
    free(kk);
    free(qq);
    free(vv);
    free(path);
    return err;
}

/*
 * The commit: state_out[b][h] = the recurrence run from state_in[b][h] over
 * acc_nodes[b][0 .. acc_len[b]) in order.  Returns 0, or -1 on an accepted
 * count or node outside the tree.
 */
int oracle_delta_commit(int dtype, int B, int N, int Hk, int Hv, int dk, int dv, const uint16_t* k,
                        const uint16_t* v, const float* alpha, const float* beta, const int32_t* acc_nodes,
                        const int32_t* acc_len, const float* state_in, double* state_out) {
    if (B < 1 || N < 1 || Hk < 1 || Hv < 1 || Hv % Hk != 0 || dk < 1 || dv < 1) return -1;
    const int G = Hv / Hk;
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    double* kk = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    int err = (!u || !kk || !vv) ? -1 : 0;
    for (int b = 0; b < B && !err; ++b) {
        const int a = acc_len[b];
        if (a < 0 || a > N) {
            err = -1;
            break;
        }
        for (int h = 0; h < Hv; ++h) {
            const size_t base = ((size_t)b * Hv + h) * (size_t)dk * dv;
            double* S = state_out + base;
            for (size_t x = 0; x < (size_t)dk * dv; ++x) S[x] = state_in[base + x];
            for (int t = 0; t < a && !err; ++t) {
                const int n = acc_nodes[(size_t)b * N + t];
                if (n < 0 || n >= N) {
                    err = -1;
                    break;
                }
                const size_t node = (size_t)b * N + n;
                delta_load(dtype, k + (node * Hk + h / G) * dk, dk, kk);
                delta_load(dtype, v + (node * Hv + h) * dv, dv, vv);
                delta_update(dk, dv, S, kk, vv, alpha[node * Hv + h], beta[node * Hv + h], u);
            }
        }
    }
    free(u);
    free(kk);
    free(vv);
    return err;
}
