"""Pins for the fp64 oracle against facts it does not compute itself: values
worked by hand, closed forms, independent textbook routines (numpy / torch
CPU), exhaustive checks of the 16-bit upcasts, and brute-force enumeration of
root paths.  Each pin targets a mistake that could plausibly hide in the
oracle (a dropped mask term, a wrong GQA head, a wrong page index, a reversed
path, a wrong tie rule)."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers

def _bits(vals, dtype):
    a = np.asarray(vals, dtype=np.float32)
    return W.f32_to_bf16_bits(a) if dtype == W.BF16 else W.f32_to_f16_bits(a)


def _hand_tree_inputs(dtype=W.F16):
    """Hand example: D=1, one head, q=1, one committed key k=0 (v=0), tree
    parent=[-1,0,0], tree keys [1, 0, 2], tree values [4, 8, -4], scale ln 2,
    so each visible key's weight is 2**k."""
    q = np.array([[[[1.0]], [[1.0]], [[1.0]]]], dtype=np.float32)  # [1][3][1][1]
    kp = np.zeros((1, 1, 64, 1), np.float32)
    vp = np.zeros((1, 1, 64, 1), np.float32)
    return dict(q=_bits(q, dtype), k_pool=_bits(kp, dtype), v_pool=_bits(vp, dtype),
                page_table=np.array([[0]], np.int32), ctx_len=np.array([1], np.int32),
                k_tree=_bits(np.array([1.0, 0.0, 2.0]).reshape(1, 3, 1, 1), dtype),
                v_tree=_bits(np.array([4.0, 8.0, -4.0]).reshape(1, 3, 1, 1), dtype),
                parent=np.array([[-1, 0, 0]], np.int32))


def _gather_logical(inp, b, g, dtype_id):
    """K, V of sequence b / kv-head g in logical order, fp64, via numpy indexing."""
    L = int(inp["ctx_len"][b])
    pos = np.arange(L)
    pages = inp["page_table"][b][pos // 64]
    slots = pos % 64
    k = inp["k_pool"][pages, g, slots, :]
    v = inp["v_pool"][pages, g, slots, :]
    return _to64(k, dtype_id), _to64(v, dtype_id)


def _to64(bits, dtype_id):
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype_id == oracle.BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


# ---------------------------------------------------------------- upcasts

def test_upcast_bf16_exhaustive():
    lib_vals = np.array([oracle.upcast(oracle.BF16, b) for b in range(65536)])
    ref = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(lib_vals), nan)
    assert np.array_equal(lib_vals[~nan], ref[~nan])


def test_upcast_f16_exhaustive():
    lib_vals = np.array([oracle.upcast(oracle.F16, b) for b in range(65536)])
    ref = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(lib_vals), nan)
    assert np.array_equal(lib_vals[~nan], ref[~nan])
    assert oracle.upcast(oracle.F16, 0x0001) == 2.0 ** -24
    assert oracle.upcast(oracle.F16, 0x7BFF) == 65504.0


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_attention_hand_example(dtype):
    inp = _hand_tree_inputs(dtype)
    did = oracle.BF16 if dtype == W.BF16 else oracle.F16
    out, lse = oracle.verify_attn(inp, did, scale=math.log(2.0), threads=1)
    # node 0 sees {prefix 1, n0 2}: 8/3; node 1 sees {1, 2, 1}: 16/4;
    # node 2 sees {1, 2, 4}: (8 - 16)/7
    np.testing.assert_allclose(out[:, 0], [8.0 / 3.0, 4.0, -8.0 / 7.0], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, [math.log(3.0), math.log(4.0), math.log(7.0)], rtol=1e-13)


def test_attention_equal_keys_is_mean_of_visible_values():
    cfg = W.TINY.replace(ctx=(200,), N=6, Hq=4, Hkv=2, D=16)
    inp = W.generate(cfg, seed=3, fill_unused="nan")
    inp["k_pool"][:] = W.f32_to_f16_bits(np.full(1, 0.5))[0]
    inp["k_tree"][:] = inp["k_pool"].flat[0]
    out, _ = oracle.verify_attn(inp, oracle.F16, threads=2)
    out = out.reshape(1, cfg.N, cfg.Hq, cfg.D)
    for h in range(cfg.Hq):
        g = h // (cfg.Hq // cfg.Hkv)
        _, vpre = _gather_logical(inp, 0, g, oracle.F16)
        vt = _to64(inp["v_tree"][0, :, g, :], oracle.F16)
        for i in range(cfg.N):
            path, c = [], i
            while c >= 0:
                path.append(c)
                c = int(inp["parent"][0, c])
            vis = np.concatenate([vpre, vt[path]], axis=0)
            np.testing.assert_allclose(out[0, i, h], vis.mean(axis=0), rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
def test_one_node_tree_is_plain_decode(dtype):
    cfg = W.VerifyConfig("decode", ctx=(300, 77), Hq=6, Hkv=2, D=32, dtype=dtype, N=1,
                         paged="permuted", spare_pages=5, vocab=64)
    inp = W.generate(cfg, seed=11)
    did = oracle.BF16 if dtype == W.BF16 else oracle.F16
    scale = 1.0 / math.sqrt(cfg.D)
    out, lse = oracle.verify_attn(inp, did, threads=2)
    out = out.reshape(cfg.B, cfg.Hq, cfg.D)
    for b in range(cfg.B):
        for h in range(cfg.Hq):
            g = h // cfg.G
            k, v = _gather_logical(inp, b, g, did)
            k = np.vstack([k, _to64(inp["k_tree"][b, 0, g], did)[None]])
            v = np.vstack([v, _to64(inp["v_tree"][b, 0, g], did)[None]])
            q = _to64(inp["q"][b, 0, h], did)
            logits = (k @ q) * scale
            w = np.exp(logits - logits.max())
            ref = (w / w.sum()) @ v
            np.testing.assert_allclose(out[b, h], ref, rtol=1e-11, atol=1e-14)
            assert abs(lse[b * cfg.Hq + h] - (logits.max() + np.log(w.sum()))) < 1e-11


def test_chain_tree_is_causal_attention():
    torch = pytest.importorskip("torch")
    cfg = W.VerifyConfig("chain", ctx=(130,), Hq=4, Hkv=1, D=16, dtype=W.BF16, N=9, tree="chain",
                         vocab=64, paged="permuted", spare_pages=3)
    inp = W.generate(cfg, seed=5)
    out, _ = oracle.verify_attn(inp, oracle.BF16, threads=2)
    out = out.reshape(cfg.N, cfg.Hq, cfg.D)
    k, v = _gather_logical(inp, 0, 0, oracle.BF16)
    kt = _to64(inp["k_tree"][0, :, 0, :], oracle.BF16)
    vt = _to64(inp["v_tree"][0, :, 0, :], oracle.BF16)
    K = torch.from_numpy(np.vstack([k, kt]))[None, None].expand(1, cfg.Hq, -1, -1)
    V = torch.from_numpy(np.vstack([v, vt]))[None, None].expand(1, cfg.Hq, -1, -1)
    Q = torch.from_numpy(_to64(inp["q"][0], oracle.BF16)).permute(1, 0, 2)[None]  # [1][Hq][N][D]
    L = cfg.ctx[0]
    mask = torch.ones(cfg.N, L + cfg.N, dtype=torch.bool)
    mask[:, L:] = torch.tril(torch.ones(cfg.N, cfg.N, dtype=torch.bool))
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-13)


def test_non_ancestor_tree_kv_does_not_change_output():
    cfg = W.TINY.replace(ctx=(150,), N=10, D=16)
    inp = W.generate(cfg, seed=8)
    base, _ = oracle.verify_attn(inp, oracle.F16, threads=2)
    anc = oracle.ancestor_matrix(inp["parent"][0])
    rng = np.random.default_rng(0)
    i = 7
    non = [j for j in range(cfg.N) if not anc[i, j]]
    assert non, "test tree should have non-ancestors of node 7"
    pert = {k: v.copy() for k, v in inp.items()}
    pert["k_tree"][0, non] = rng.integers(0, 0x3C00, size=pert["k_tree"][0, non].shape, dtype=np.uint16)
    pert["v_tree"][0, non] = rng.integers(0, 0x3C00, size=pert["v_tree"][0, non].shape, dtype=np.uint16)
    out, _ = oracle.verify_attn(pert, oracle.F16, threads=2)
    rows = slice(i * cfg.Hq, (i + 1) * cfg.Hq)
    assert np.array_equal(out[rows], base[rows])
    # and nodes that do see a perturbed node change
    seen = [r for r in range(cfg.N) if any(anc[r, j] for j in non)]
    assert any(not np.array_equal(out[r * cfg.Hq:(r + 1) * cfg.Hq], base[r * cfg.Hq:(r + 1) * cfg.Hq])
               for r in seen)


def test_page_relabelling_is_invisible():
    cfg = W.TINY.replace(ctx=(333, 64, 5), N=5, D=16, paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=9, fill_unused="random")
    base, _ = oracle.verify_attn(inp, oracle.F16, threads=2)
    perm = np.random.default_rng(1).permutation(inp["k_pool"].shape[0])
    moved = dict(inp)
    moved["k_pool"] = np.empty_like(inp["k_pool"])
    moved["v_pool"] = np.empty_like(inp["v_pool"])
    moved["k_pool"][perm] = inp["k_pool"]
    moved["v_pool"][perm] = inp["v_pool"]
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    moved["page_table"] = pt
    out, _ = oracle.verify_attn(moved, oracle.F16, threads=2)
    assert np.array_equal(out, base)


def test_empty_prefix_sees_only_tree():
    inp = _hand_tree_inputs()
    inp["ctx_len"] = np.array([0], np.int32)
    out, _ = oracle.verify_attn(inp, oracle.F16, scale=math.log(2.0), threads=1)
    # node 0 sees only itself: 4; node 1 {2,1}: (8+8)/3; node 2 {2,4}: (8-16)/6
    np.testing.assert_allclose(out[:, 0], [4.0, 16.0 / 3.0, -8.0 / 6.0], rtol=1e-13)


def test_ancestor_matrix_hand():
    anc = oracle.ancestor_matrix(np.array([-1, 0, 0, 1, 3], np.int32))
    exp = np.array([[1, 0, 0, 0, 0],
                    [1, 1, 0, 0, 0],
                    [1, 0, 1, 0, 0],
                    [1, 1, 0, 1, 0],
                    [1, 1, 0, 1, 1]], np.uint8)
    assert np.array_equal(anc, exp)


# ---------------------------------------------------------------- argmax

def test_argmax_matches_numpy_first_index_with_ties_and_zeros():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 1000)).astype(np.float32)
    x[1, 10] = x[1, 500] = 99.0            # tie: lowest index wins
    x[2, :] = 0.0
    x[2, 3] = -0.0                         # -0.0 ties +0.0
    x[3, :] = -0.0
    x[3, 7] = 0.0
    x[4, -1] = 50.0                        # maximum at the last index
    x[5, :] = -np.inf
    x[6, :] = 7.0
    assert np.array_equal(oracle.argmax(x), np.argmax(x, axis=1).astype(np.int32))
    assert oracle.argmax(x)[1] == 10
    assert oracle.argmax(x)[2] == 0


# ---------------------------------------------------------------- acceptance

def _paths_top_down(parent):
    """Every root path, built from the root downward over child lists."""
    n = len(parent)
    kids = {-1: []}
    for i in range(n):
        kids.setdefault(int(parent[i]), []).append(i)
    out, stack = [], [[]]
    while stack:
        path = stack.pop()
        last = path[-1] if path else -1
        for c in kids.get(last, []):
            stack.append(path + [c])
            out.append(path + [c])
    return out


def _brute_accept(parent, draft, am):
    best = []
    for path in _paths_top_down(parent):
        rows = [0] + [c + 1 for c in path[:-1]]
        if all(draft[c] == am[r] for c, r in zip(path, rows)):
            if len(path) > len(best) or (len(path) == len(best) and path[-1] < best[-1]):
                best = path
    bonus = am[best[-1] + 1] if best else am[0]
    return best, bonus


def test_accept_hand_example():
    acc, alen, bonus = oracle.accept(np.array([[-1, 0, 0]]), np.array([[5, 7, 9]]), np.array([[5, 9, 3, 4]]))
    assert alen[0] == 2 and list(acc[0, :2]) == [0, 2] and bonus[0] == 4
    assert acc[0, 2] == -1
    acc, alen, bonus = oracle.accept(np.array([[-1, 0, 0]]), np.array([[6, 7, 9]]), np.array([[5, 9, 3, 4]]))
    assert alen[0] == 0 and bonus[0] == 5


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7])
def test_accept_brute_force_random_trees(n):
    rng = np.random.default_rng(100 + n)
    B = 10000
    vocab = 3  # tiny vocabulary: many matches, duplicate sibling tokens included
    parent = np.zeros((B, n), np.int32)
    for b in range(B):
        parent[b, 0] = -1 if rng.random() < 0.8 else -1
        for i in range(1, n):
            parent[b, i] = rng.integers(-1, i)
    draft = rng.integers(0, vocab, size=(B, n)).astype(np.int32)
    am = rng.integers(0, vocab, size=(B, n + 1)).astype(np.int32)
    acc, alen, bonus = oracle.accept(parent, draft, am)
    for b in range(0, B, 7 if n > 5 else 1):
        path, bo = _brute_accept(parent[b], draft[b], am[b])
        assert alen[b] == len(path)
        assert list(acc[b, :alen[b]]) == path
        assert bonus[b] == bo


def test_accept_greedy_walk_for_distinct_siblings():
    """With distinct sibling tokens the deepest matching path is the greedy walk
    down from the root."""
    cfg = W.GQA27B_32K.replace(ctx=(64,), vocab=50, N=22)
    for seed in range(200):
        rng = np.random.default_rng(seed)
        par = W.random_parents(rng, cfg.N, "random", 4)
        dr = W.draft_tokens(rng, par, cfg.vocab)
        lg = W.planted_logits(rng, par, dr, cfg.vocab, 0.9)
        am = np.argmax(lg, axis=1).astype(np.int32)
        acc, alen, bonus = oracle.accept(par[None], dr[None], am[None])
        walk, cur = [], -1
        while True:
            t = am[cur + 1]
            nxt = [c for c in range(cfg.N) if par[c] == cur and dr[c] == t]
            if not nxt:
                break
            cur = nxt[0]
            walk.append(cur)
        assert list(acc[0, :alen[0]]) == walk
        assert bonus[0] == am[walk[-1] + 1 if walk else 0]


def test_accept_chain_full_plant_accepts_everything():
    n = 12
    par = np.arange(-1, n - 1, dtype=np.int32)[None]
    dr = np.arange(100, 100 + n, dtype=np.int32)[None]
    am = np.concatenate([dr[0], [7]]).astype(np.int32)[None]
    acc, alen, bonus = oracle.accept(par, dr, am)
    assert alen[0] == n and list(acc[0]) == list(range(n)) and bonus[0] == 7


def test_accept_result_is_prefix_closed_root_path():
    rng = np.random.default_rng(4)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        par = W.random_parents(rng, n, "random", 4)
        dr = W.draft_tokens(rng, par, 6)
        am = rng.integers(0, 6, size=n + 1).astype(np.int32)
        acc, alen, _ = oracle.accept(par[None], dr[None], am[None])
        path = list(acc[0, :alen[0]])
        prev = -1
        for c in path:
            assert par[c] == prev
            prev = c
        assert all(x == -1 for x in acc[0, alen[0]:])


def test_accept_rejects_non_topological_parent():
    with pytest.raises(ValueError):
        oracle.accept(np.array([[-1, 2, 0]]), np.array([[1, 2, 3]]), np.array([[1, 2, 3, 4]]))


# ---------------------------------------------------------------- commit

def test_commit_hand_example():
    cfg = W.TINY.replace(ctx=(64,), N=3, Hq=2, Hkv=1, D=8, paged="permuted", spare_pages=2)
    inp = W.generate(cfg, seed=1)
    acc = np.array([[0, 2, -1]], np.int32)
    kp, vp, ctx = oracle.commit(inp, acc, np.array([2], np.int32))
    page = inp["page_table"][0, 1]
    assert ctx[0] == 66
    assert np.array_equal(kp[page, 0, 0], inp["k_tree"][0, 0, 0])
    assert np.array_equal(kp[page, 0, 1], inp["k_tree"][0, 2, 0])
    assert np.array_equal(vp[page, 0, 1], inp["v_tree"][0, 2, 0])
    # every other byte is unchanged
    mask = np.ones(kp.shape[:3], bool)
    mask[page, 0, 0:2] = False
    assert np.array_equal(kp[mask], inp["k_pool"][mask])
    assert np.array_equal(vp[mask], inp["v_pool"][mask])


def test_commit_then_verify_equals_extended_prefix():
    """After committing the accepted path, the committed prefix attends exactly
    like a prefix that had those tokens all along."""
    cfg = W.TINY.replace(ctx=(70, 128), N=6, D=16, paged="permuted", spare_pages=3)
    inp = W.generate(cfg, seed=12)
    acc = np.full((2, 6), -1, np.int32)
    acc[0, :2] = [0, 3]
    acc[1, :1] = [0]
    kp, vp, ctx = oracle.commit(inp, acc, np.array([2, 1], np.int32))
    for b in range(2):
        L = int(inp["ctx_len"][b])
        pos = np.arange(L, int(ctx[b]))
        pages = inp["page_table"][b][pos // 64]
        got = kp[pages, :, pos % 64, :]
        want = inp["k_tree"][b, acc[b, :len(pos)]]
        assert np.array_equal(got, want)


# ---------------------------------------------------------------- lm_head + argmax

def _bits_to_f64(bits, dtype):
    """Independent upcast through numpy's own float formats."""
    bits = np.asarray(bits, np.uint16)
    if dtype == oracle.BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def test_lmhead_hand_example_ties_across_slices():
    # hidden [1,0] / [0,1]; weight rows [1,0] [2,0] [0,3] [2,0] (bf16 bits)
    h = np.array([[0x3F80, 0x0000], [0x0000, 0x3F80]], np.uint16)
    w = np.array([[0x3F80, 0], [0x4000, 0], [0, 0x4040], [0x4000, 0]], np.uint16)
    for threads in (1, 2, 3, 4):
        idx, top1, top2 = oracle.lmhead_argmax(h, w, oracle.BF16, threads=threads)
        # row 0: logits [1, 2, 0, 2] -> the tie between 1 and 3 goes to 1; second best is the tied 2
        # row 1: logits [0, 0, 3, 0]
        assert idx.tolist() == [1, 2]
        assert top1.tolist() == [2.0, 3.0]
        assert top2.tolist() == [2.0, 0.0]


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.F16])
def test_lmhead_matches_numpy_matmul_argmax(dtype):
    rng = np.random.default_rng(5)
    rows, d_model, vocab = 9, 96, 1500
    hf = rng.standard_normal((rows, d_model)).astype(np.float32)
    wf = (0.05 * rng.standard_normal((vocab, d_model))).astype(np.float32)
    if dtype == oracle.BF16:
        hb, wb = W.f32_to_bf16_bits(hf), W.f32_to_bf16_bits(wf)
    else:
        hb, wb = W.f32_to_f16_bits(hf), W.f32_to_f16_bits(wf)
    # a planted exact tie: row 2's best entry duplicated at a higher index
    logits0 = _bits_to_f64(hb, dtype) @ _bits_to_f64(wb, dtype).T
    best = int(np.argmax(logits0[2]))
    wb[vocab - 1] = wb[best]
    logits = _bits_to_f64(hb, dtype) @ _bits_to_f64(wb, dtype).T
    idx, top1, top2 = oracle.lmhead_argmax(hb, wb, dtype, threads=5)
    assert idx.tolist() == np.argmax(logits, axis=1).tolist()
    srt = np.sort(logits, axis=1)
    assert np.allclose(top1, srt[:, -1], rtol=1e-12, atol=1e-12)
    assert np.allclose(top2, srt[:, -2], rtol=1e-12, atol=1e-12)
    assert top1[2] == top2[2]  # the planted tie


def test_lmhead_thread_count_does_not_change_the_result():
    rng = np.random.default_rng(6)
    hb = W.f32_to_bf16_bits(rng.standard_normal((5, 64)).astype(np.float32))
    wb = W.f32_to_bf16_bits(rng.standard_normal((777, 64)).astype(np.float32))
    ref = oracle.lmhead_argmax(hb, wb, oracle.BF16, threads=1)
    for t in (2, 7, 64):
        got = oracle.lmhead_argmax(hb, wb, oracle.BF16, threads=t)
        assert all(np.array_equal(a, b) for a, b in zip(ref, got))


# ---------------------------------------------------------------- gated delta rule (tree-aware recurrent state)

def _f16(x):
    return np.asarray(x, np.float16).view(np.uint16)


def _delta_case(q, k, v, alpha, beta, parent, state):
    """One sequence, one key head, one value head: q, k [N][dk], v [N][dv]."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    N = q.shape[0]
    return dict(q=_f16(q).reshape(1, N, 1, -1), k=_f16(k).reshape(1, N, 1, -1), v=_f16(v).reshape(1, N, 1, -1),
                alpha=np.asarray(alpha, np.float32).reshape(1, N, 1), beta=np.asarray(beta, np.float32).reshape(1, N, 1),
                parent=np.asarray(parent, np.int32).reshape(1, N),
                state=np.asarray(state, np.float32).reshape(1, 1, q.shape[1], v.shape[1]))


def test_delta_hand_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "delta_rule_hand_example.json")))
    inp = _delta_case(g["q"], g["k"], g["v"], g["alpha"], g["beta"], g["parent"], g["state"])
    out = oracle.delta_tree(inp, oracle.F16)[0, :, 0, :]
    assert np.array_equal(out, np.asarray(g["out"], np.float64))
    N = len(g["parent"])
    for c in g["commits"]:
        path = c["path"]
        acc = np.full((1, N), -1, np.int32)
        acc[0, :len(path)] = path
        st = oracle.delta_commit(inp, oracle.F16, acc, np.array([len(path)], np.int32))[0, 0]
        assert np.array_equal(st, np.asarray(c["state"], np.float64)), path


def test_delta_no_write_no_decay_is_a_matrix_vector_product():
    cfg = W.DeltaConfig("pin-nowrite", B=2, N=9, Hk=2, Hv=4, dk=16, dv=8, dtype=W.F16)
    inp = W.generate_delta(cfg, seed=3)
    inp["beta"][:] = 0.0
    inp["alpha"][:] = 1.0
    out = oracle.delta_tree(inp, oracle.F16)
    q = inp["q"].view(np.float16).astype(np.float64)
    for b in range(2):
        for h in range(4):
            ref = q[b, :, h // 2, :] @ inp["state"][b, h].astype(np.float64)
            assert np.allclose(out[b, :, h, :], ref, rtol=1e-12, atol=1e-12)


def test_delta_pure_decay_multiplies_the_path_gates():
    cfg = W.DeltaConfig("pin-decay", B=1, N=12, Hk=1, Hv=2, dk=8, dv=8, dtype=W.F16, tree="random", branch_cap=3)
    inp = W.generate_delta(cfg, seed=4)
    inp["beta"][:] = 0.0
    out = oracle.delta_tree(inp, oracle.F16)
    anc = oracle.ancestor_matrix(inp["parent"][0])  # anc[i][j]: j is i or an ancestor of i
    q = inp["q"].view(np.float16).astype(np.float64)
    for h in range(2):
        base = q[0, :, 0, :] @ inp["state"][0, h].astype(np.float64)
        gate = np.array([np.prod(inp["alpha"][0, anc[i].astype(bool), h].astype(np.float64)) for i in range(12)])
        assert np.allclose(out[0, :, h, :], gate[:, None] * base, rtol=1e-12, atol=1e-14)


def test_delta_full_write_at_a_basis_key_reads_back_the_value():
    # beta = 1 and k = e_m replace row m of the state by v (whatever alpha is),
    # so reading with q = e_m returns v exactly
    cfg = W.DeltaConfig("pin-write", B=1, N=16, Hk=1, Hv=1, dk=8, dv=8, dtype=W.F16, tree="random", branch_cap=2)
    inp = W.generate_delta(cfg, seed=5)
    rng = np.random.default_rng(5)
    m = rng.integers(0, 8, size=16)
    e = np.zeros((16, 8))
    e[np.arange(16), m] = 1.0
    inp["k"][0, :, 0, :] = _f16(e)
    inp["q"][0, :, 0, :] = _f16(e)
    inp["beta"][:] = 1.0
    out = oracle.delta_tree(inp, oracle.F16)[0, :, 0, :]
    assert np.array_equal(out, inp["v"][0, :, 0, :].view(np.float16).astype(np.float64))


def test_delta_relabelling_the_tree_permutes_the_outputs():
    cfg = W.DeltaConfig("pin-relabel", B=1, N=10, Hk=1, Hv=2, dk=8, dv=4, dtype=W.F16, tree="random", branch_cap=3)
    inp = W.generate_delta(cfg, seed=6)
    par = inp["parent"][0]
    # another topological order: by depth, then by reversed index
    depth = np.zeros(10, int)
    for i in range(10):
        depth[i] = 0 if par[i] < 0 else depth[par[i]] + 1
    order = sorted(range(10), key=lambda i: (depth[i], -i))
    new_of = {old: new for new, old in enumerate(order)}
    p2 = np.array([-1 if par[o] < 0 else new_of[par[o]] for o in order], np.int32)
    inp2 = dict(inp)
    for key in ("q", "k", "v", "alpha", "beta"):
        inp2[key] = np.ascontiguousarray(inp[key][:, order])
    inp2["parent"] = p2[None, :]
    a = oracle.delta_tree(inp, oracle.F16)
    b = oracle.delta_tree(inp2, oracle.F16)
    assert np.array_equal(a[:, order], b)


def test_delta_commit_reads_back_the_node_output_and_empty_commit_keeps_the_state():
    cfg = W.DeltaConfig("pin-commit", B=2, N=12, Hk=1, Hv=2, dk=8, dv=8, dtype=W.F16, tree="random", branch_cap=3)
    inp = W.generate_delta(cfg, seed=7)
    out = oracle.delta_tree(inp, oracle.F16)
    q = inp["q"].view(np.float16).astype(np.float64)
    for i in range(12):
        acc = np.full((2, 12), -1, np.int32)
        lens = np.zeros(2, np.int32)
        for b in range(2):
            anc = oracle.ancestor_matrix(inp["parent"][b])
            path = [j for j in range(12) if anc[i, j]]  # ancestors in index order = root-to-leaf
            acc[b, :len(path)] = path
            lens[b] = len(path)
        st = oracle.delta_commit(inp, oracle.F16, acc, lens)
        for b in range(2):
            for h in range(2):
                assert np.allclose(q[b, i, 0] @ st[b, h], out[b, i, h], rtol=1e-12, atol=1e-13)
    none = oracle.delta_commit(inp, oracle.F16, np.zeros((2, 12), np.int32), np.zeros(2, np.int32))
    assert np.array_equal(none, inp["state"].astype(np.float64))


def test_delta_rejects_a_bad_parent():
    inp = W.generate_delta(W.DeltaConfig("pin-bad", N=4, Hk=1, Hv=1, dk=4, dv=4, dtype=W.F16), seed=1)
    inp["parent"] = np.array([[-1, 0, 3, 1]], np.int32)
    with pytest.raises(ValueError):
        oracle.delta_tree(inp, oracle.F16)


# ---------------------------------------------------------------- host-resident pages

def test_stage_pages_hand_example():
    host_k = np.arange(3 * 2, dtype=np.uint16).reshape(3, 2) + 100   # 3 host pages of 2 values
    host_v = host_k + 1000
    pool_k = np.zeros((4, 2), np.uint16)
    pool_v = np.zeros((4, 2), np.uint16)
    table = np.array([[0, -1, 3], [1, -1, -1]], np.int32)
    kp, vp, pt = oracle.stage_pages(host_k, host_v, [2, 0], [1, 2], pool_k, pool_v, table_idx=[1, 4],
                                    page_table=table)
    assert kp.tolist() == [[0, 0], [104, 105], [100, 101], [0, 0]]
    assert vp.tolist() == [[0, 0], [1104, 1105], [1100, 1101], [0, 0]]
    assert pt.tolist() == [[0, 1, 3], [1, 2, -1]]
    assert pool_k.sum() == 0 and table[0, 1] == -1  # inputs untouched


# ---------------------------------------------------------------- quantised V storage

def test_dequant_v_hand_examples():
    # int8: codes 3, -5, 127 at exponents 127 (x1), 126 (x1/2), 0 (zero)
    codes = np.array([[3, 0xFB], [127, 1], [7, 7]], np.uint8)[None]     # [1][3 tokens][2 dims]
    exps = np.array([[127, 126, 0]], np.uint8)
    got = oracle.dequant_v(codes, exps, oracle.V_INT8, oracle.F16).view(np.float16).astype(float)
    assert got.tolist() == [[[3.0, -5.0], [63.5, 0.5], [0.0, 0.0]]]
    # int4: byte 0x9F holds even dim 0xF = -1 and odd dim 0x9 = -7; byte 0x71 holds 1 and 7
    codes4 = np.array([[[0x9F, 0x71]]], np.uint8)                      # [1][1 token][4 dims]
    got4 = oracle.dequant_v(codes4, np.array([[129]], np.uint8), oracle.V_INT4, oracle.BF16)
    vals = (got4.astype(np.uint32) << 16).view(np.float32).astype(float)
    assert vals.tolist() == [[[-4.0, -28.0, 4.0, 28.0]]]


def test_dequant_v_is_exact_over_the_code_and_exponent_range():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(2, 64, 16)).astype(np.uint8)
    exps = rng.integers(103, 136, size=(2, 64)).astype(np.uint8)
    for dt in (oracle.F16, oracle.BF16):
        oracle.dequant_v(codes, exps, oracle.V_INT8, dt)  # raises if any value were rounded
    with pytest.raises(ValueError):  # 127 * 2^9 = 65024 is still fp16, 127 * 2^10 is not
        oracle.dequant_v(np.full((1, 1, 2), 127, np.uint8), np.array([[137]], np.uint8), oracle.V_INT8, oracle.F16)


# ---------------------------------------------------------------- quantised K storage (FP8 E4M3 codes)

def test_decode_e4m3_matches_torch_on_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_e4m3_hand_values_and_dequant():
    got = oracle.decode_e4m3([0x38, 0x7E, 0x01, 0xB8, 0x00, 0x80, 0x3C])
    assert got.tolist() == [1.0, 448.0, 2.0 ** -9, -1.0, 0.0, -0.0, 1.5]
    # code 1.5 at exponent 126 (x 1/2) -> 0.75; exponent 0 -> 0
    bits = oracle.dequant_k_e4m3(np.array([[[0x3C, 0xB8]]], np.uint8), np.array([[126]], np.uint8), oracle.F16)
    assert bits.view(np.float16).astype(float).tolist() == [[[0.75, -0.5]]]
    zero = oracle.dequant_k_e4m3(np.array([[[0x3C]]], np.uint8), np.array([[0]], np.uint8), oracle.BF16)
    assert zero.tolist() == [[[0]]]
    with pytest.raises(ValueError):
        oracle.dequant_k_e4m3(np.array([[[0x7F]]], np.uint8), np.array([[127]], np.uint8), oracle.F16)


def _bf16_bits(vals):
    return W.f32_to_bf16_bits(np.asarray(vals, np.float32))


def test_quantise_k_hand_rows():
    # max 1 -> p = 8 (256 <= 448 < 512), e = 119; codes of 256, -128, 0 and 0.75
    codes, e = oracle.quantise_k_e4m3(_bf16_bits([[1.0, -0.5, 0.0, 3.0 * 2.0 ** -10]]), oracle.BF16)
    assert e.tolist() == [119] and codes.tolist() == [[0x78, 0xF0, 0x00, 0x34]]
    # max 448 -> p = 0; 272 and 304 lie halfway between neighbours and go to the even code
    codes, e = oracle.quantise_k_e4m3(_bf16_bits([[448.0, 272.0, 304.0, -272.0]]), oracle.BF16)
    assert e.tolist() == [127] and codes.tolist() == [[0x7E, 0x78, 0x7A, 0xF8]]
    # an all-zero row
    codes, e = oracle.quantise_k_e4m3(np.zeros((1, 4), np.uint16), oracle.F16)
    assert e.tolist() == [0] and codes.tolist() == [[0, 0, 0, 0]]


def test_quantise_k_matches_torch_rounding_and_scale_rule():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(8)
    k = W.f32_to_bf16_bits(rng.standard_normal((300, 256)).astype(np.float32) * np.float32(3.0))
    codes, e = oracle.quantise_k_e4m3(k, oracle.BF16)
    x = oracle._bits_to_f64(k, oracle.BF16)
    p = 127 - e.astype(np.int64)
    y = x * np.ldexp(1.0, p)[:, None]                       # exact in float32 (bf16 times a power of two)
    m = np.abs(y).max(axis=1)
    assert (m > 224).all() and (m <= 448).all()             # the row maximum lands in (224, 448]
    ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_quantise_then_dequantise_error_and_fixed_points():
    rng = np.random.default_rng(9)
    k = W.f32_to_bf16_bits(rng.standard_normal((200, 128)).astype(np.float32))
    codes, e = oracle.quantise_k_e4m3(k, oracle.BF16)
    back = oracle._bits_to_f64(oracle.dequant_k_e4m3(codes[:, None, :], e[:, None], oracle.BF16)[:, 0, :],
                               oracle.BF16)
    x = oracle._bits_to_f64(k, oracle.BF16)
    step = np.ldexp(1.0, 127 - e.astype(np.int64) - 9)[:, None]   # E4M3's subnormal step at the row's scale
    assert (np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, step / 2)).all()
    # values already of the form e4m3(code) * 2^(e - 127) come back unchanged
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    c0 = finite[rng.integers(0, len(finite), size=(50, 64))]
    e0 = rng.integers(118, 126, size=50).astype(np.uint8)
    v = oracle.dequant_k_e4m3(c0[:, None, :], e0[:, None], oracle.BF16)[:, 0, :]
    c1, e1 = oracle.quantise_k_e4m3(v, oracle.BF16)
    assert np.array_equal(oracle.dequant_k_e4m3(c1[:, None, :], e1[:, None], oracle.BF16)[:, 0, :], v)


def test_commit_kq_hand_example():
    """L = 64, accepted path [0, 2] of a 3-node tree, one KV head, D = 4: node
    0's K row lands in page_table[0][1] slot 0 and node 2's in slot 1, each as
    the quantised row worked by hand (see test_quantise_k_hand_rows); every
    other byte keeps its value."""
    kt = np.zeros((1, 3, 1, 4), np.uint16)
    kt[0, 0, 0] = _bf16_bits([1.0, -0.5, 0.0, 3.0 * 2.0 ** -10])    # e 119, codes 78 F0 00 34
    kt[0, 1, 0] = _bf16_bits([5.0, 5.0, 5.0, 5.0])                   # rejected: never written
    kt[0, 2, 0] = _bf16_bits([448.0, 272.0, 304.0, -272.0])          # e 127, codes 7E 78 7A F8
    inp = dict(k_tree=kt, page_table=np.array([[3, 1, 0, 2]], np.int32), ctx_len=np.array([64], np.int32),
               dtype_id=oracle.BF16)
    codes = np.full((4, 1, 64, 4), 0x11, np.uint8)
    expo = np.full((4, 1, 64), 0x22, np.uint8)
    c, e = oracle.commit_kq(inp, codes, expo, np.array([[0, 2, -1]], np.int32), np.array([2], np.int32))
    assert c[1, 0, 0].tolist() == [0x78, 0xF0, 0x00, 0x34] and e[1, 0, 0] == 119
    assert c[1, 0, 1].tolist() == [0x7E, 0x78, 0x7A, 0xF8] and e[1, 0, 1] == 127
    untouched = np.ones(codes.shape[:3], bool)
    untouched[1, 0, :2] = False
    assert (c[untouched] == 0x11).all() and (e[untouched] == 0x22).all()
    assert (codes == 0x11).all() and (expo == 0x22).all()  # not in place: the inputs are left alone


def test_commit_kq_touches_the_rows_the_16bit_commit_touches():
    """On a ragged 3-sequence batch, the rows commit_kq writes are exactly the
    rows the 16-bit commit writes, and each reads back (dequant_k_e4m3) as the
    quantised form of the accepted node's K row."""
    cfg = W.VerifyConfig("commit-kq", ctx=(64, 130, 1000), Hq=4, Hkv=2, D=128, dtype=W.BF16, N=10,
                         tree="random", vocab=8, p_plant=0.95, paged="permuted", spare_pages=3)
    inp = W.generate(cfg, seed=2)
    am = oracle.argmax(inp["logits"])
    acc, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    assert alen.sum() >= 3
    kq = W.generate_kq(cfg, seed=2)
    c, e = oracle.commit_kq(dict(inp, dtype_id=oracle.BF16), kq["k_codes"], kq["k_exp"], acc, alen)
    kp, _, _ = oracle.commit(inp, acc, alen)
    changed16 = (kp != inp["k_pool"]).any(axis=-1) | np.zeros(kp.shape[:3], bool)
    # rows of the 16-bit pool may be unchanged by chance only if the tree row equals the old row: never here
    changed_kq = (c != kq["k_codes"]).any(axis=-1) | (e != kq["k_exp"])
    assert np.array_equal(changed_kq, changed16)
    for b in range(cfg.B):
        for k in range(int(alen[b])):
            pos = int(inp["ctx_len"][b]) + k
            page = int(inp["page_table"][b, pos // 64])
            want_c, want_e = oracle.quantise_k_e4m3(inp["k_tree"][b, acc[b, k]], oracle.BF16)
            assert np.array_equal(c[page, :, pos % 64], want_c) and np.array_equal(e[page, :, pos % 64], want_e)
