"""Ancestor masks, argmax, acceptance and commit through the C-ABI: bit-exact
against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import bits16, cached_inputs, to_device

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _status():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------- ancestor masks

def test_anc_mask_matches_oracle_ancestors(cuda_dev):
    import torch
    LT = _lt()
    rng = np.random.default_rng(0)
    for n in (1, 2, 7, 22, 40, 63, 64):
        par = np.stack([W.random_parents(rng, n, "random", None if b % 2 else 4) for b in range(32)])
        anc = torch.empty(32, n, dtype=torch.int64, device="cuda")
        st = _status()
        LT.lucetree_build_anc_mask(_t(par), anc, st)
        bits = anc.cpu().numpy().view(np.uint64)
        assert st.item() == 0
        for b in range(32):
            ref = oracle.ancestor_matrix(par[b])
            got = ((bits[b][:, None] >> np.arange(n, dtype=np.uint64)[None, :]) & np.uint64(1)).astype(np.uint8)
            assert np.array_equal(got, ref)


def test_anc_mask_flags_bad_parent(cuda_dev):
    import torch
    LT = _lt()
    anc = torch.empty(1, 3, dtype=torch.int64, device="cuda")
    st = _status()
    LT.lucetree_build_anc_mask(_t(np.array([[-1, 2, 0]], np.int32)), anc, st)
    assert st.item() & LT.DEV_BAD_PARENT


# ---------------------------------------------------------------- argmax

def _gpu_argmax(x):
    import torch
    LT = _lt()
    rows = int(np.prod(x.shape[:-1]))
    ws = torch.empty(LT.lucetree_argmax_workspace(rows, x.shape[-1]), dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)
    out = torch.full(x.shape[:-1], -7, dtype=torch.int32, device="cuda")
    LT.lucetree_argmax(_t(x), out, ws)
    return out.cpu().numpy()


def test_argmax_planted_logits_full_vocab(cuda_dev):
    inp = W.generate(W.GQA27B_32K, with_pools=False)
    assert np.array_equal(_gpu_argmax(inp["logits"]), oracle.argmax(inp["logits"]))


@pytest.mark.parametrize("vocab", [1, 7, 1000, 1023, 4096, 151936])
def test_argmax_ties_zeros_infinities(cuda_dev, vocab):
    rng = np.random.default_rng(vocab)
    x = rng.standard_normal((41, vocab)).astype(np.float32)
    x[0, :] = 3.0                       # all equal -> index 0
    x[1, :] = -0.0
    x[1, vocab // 2] = 0.0              # -0.0 and +0.0 tie -> index 0
    x[2, :] = -np.inf
    x[3, -1] = 1e30                     # last index
    if vocab > 3:
        x[4, [vocab - 1, 2, vocab // 2]] = 77.0  # three-way tie -> 2
    x[5, :] = np.float32(-1e-45)        # denormals
    got = _gpu_argmax(x)
    assert np.array_equal(got, oracle.argmax(x))
    assert np.array_equal(got, np.argmax(x, axis=1))


def test_argmax_repeated_calls_reuse_workspace(cuda_dev):
    import torch
    LT = _lt()
    rng = np.random.default_rng(3)
    x = rng.standard_normal((23, 151936)).astype(np.float32)
    ws = torch.empty(LT.lucetree_argmax_workspace(23, 151936), dtype=torch.uint8, device="cuda")
    out = torch.empty(23, dtype=torch.int32, device="cuda")
    xt = _t(x)
    for _ in range(3):
        LT.lucetree_argmax(xt, out, ws)
        assert np.array_equal(out.cpu().numpy(), oracle.argmax(x))


# ---------------------------------------------------------------- acceptance

def _gpu_accept(par, dr, am, vocab):
    import torch
    LT = _lt()
    B, N = par.shape
    acc = torch.full((B, N), -9, dtype=torch.int32, device="cuda")
    alen = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    bonus = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    st = _status()
    LT.lucetree_accept(_t(par), _t(dr), _t(am), vocab, acc, alen, bonus, st)
    return acc.cpu().numpy(), alen.cpu().numpy(), bonus.cpu().numpy(), st.item()


@pytest.mark.parametrize("n", [1, 2, 3, 5, 7])
def test_accept_random_tiny_trees_with_duplicates(cuda_dev, n):
    rng = np.random.default_rng(n)
    B = 10000
    par = np.stack([np.array([-1] + [rng.integers(-1, i) for i in range(1, n)], np.int32) for _ in range(B)])
    dr = rng.integers(0, 3, size=(B, n)).astype(np.int32)
    am = rng.integers(0, 3, size=(B, n + 1)).astype(np.int32)
    acc, alen, bonus, st = _gpu_accept(par, dr, am, 3)
    racc, ralen, rbonus = oracle.accept(par, dr, am)
    assert st == 0
    assert np.array_equal(acc, racc) and np.array_equal(alen, ralen) and np.array_equal(bonus, rbonus)


def test_accept_every_sweep_point(cuda_dev):
    for cfg in W.sweep_points():
        inp = W.generate(cfg, seed=1, with_pools=False)
        am = oracle.argmax(inp["logits"])
        acc, alen, bonus, st = _gpu_accept(inp["parent"], inp["draft"], am, cfg.vocab)
        racc, ralen, rbonus = oracle.accept(inp["parent"], inp["draft"], am)
        assert st == 0
        assert np.array_equal(acc, racc), cfg.name
        assert np.array_equal(alen, ralen) and np.array_equal(bonus, rbonus)


def test_accept_bad_inputs_flagged(cuda_dev):
    LT = _lt()
    acc, alen, bonus, st = _gpu_accept(np.array([[-1, 1]], np.int32), np.array([[1, 2]], np.int32),
                                       np.array([[1, 2, 3]], np.int32), 10)
    assert st & LT.DEV_BAD_PARENT and alen[0] == 0 and bonus[0] == 1
    acc, alen, bonus, st = _gpu_accept(np.array([[-1, 0]], np.int32), np.array([[1, 99]], np.int32),
                                       np.array([[1, 99, 3]], np.int32), 10)
    assert st & LT.DEV_BAD_TOKEN and alen[0] == 1


# ---------------------------------------------------------------- commit

def _gpu_commit(inp, cfg, acc, alen, alias=False):
    import torch
    LT = _lt()
    d = to_device(inp, cfg)
    ctx_out = d["ctx_len"] if alias else torch.empty_like(d["ctx_len"])
    st = _status()
    LT.lucetree_commit(d["k_tree"], d["v_tree"], _t(acc), _t(alen), d["page_table"], d["ctx_len"], ctx_out,
                       d["k_pool"], d["v_pool"], st)
    torch.cuda.synchronize()
    return d, ctx_out, st.item()


@pytest.mark.parametrize("alias", [False, True])
def test_commit_small_full_pool_compare(cuda_dev, alias):
    cfg = W.VerifyConfig("commit", ctx=(64, 130, 0, 1000), Hq=4, Hkv=2, D=128, dtype=W.F16, N=12,
                         tree="random", vocab=8, p_plant=0.95, paged="permuted", spare_pages=3)
    inp = W.generate(cfg, seed=2)
    am = oracle.argmax(inp["logits"])
    acc, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    kp, vp, ctx = oracle.commit(inp, acc, alen)
    d, ctx_out, st = _gpu_commit(inp, cfg, acc, alen, alias)
    assert st == 0
    assert np.array_equal(ctx_out.cpu().numpy(), ctx)
    assert np.array_equal(bits16(d["k_pool"]), kp)
    assert np.array_equal(bits16(d["v_pool"]), vp)


@pytest.mark.slow
def test_commit_paged_256k(cuda_dev):
    import torch
    cfg = W.PAGED_256K
    inp = cached_inputs(cfg)
    # accept a full root path of the tree so the copy spans the reserved pages
    par = inp["parent"][0]
    leaf = max(range(cfg.N), key=lambda i: (len(_path(par, i)), -i))
    path = _path(par, leaf)
    acc = np.full((1, cfg.N), -1, np.int32)
    acc[0, :len(path)] = path
    alen = np.array([len(path)], np.int32)
    kp, vp, ctx = oracle.commit(inp, acc, alen)
    before_k = torch.from_numpy(inp["k_pool"].view(np.int16)).cuda()
    d, ctx_out, st = _gpu_commit(inp, cfg, acc, alen)
    assert st == 0 and ctx_out.item() == ctx[0]
    after = d["k_pool"].view(torch.int16)
    changed = (after != before_k).reshape(after.shape[0], cfg.Hkv, 64, cfg.D).any(dim=-1).nonzero().cpu().numpy()
    ref_changed = np.argwhere((kp != inp["k_pool"]).any(axis=-1))
    assert np.array_equal(changed, ref_changed)
    pages = np.unique(inp["page_table"][0, (cfg.ctx[0]) // 64:])
    pages = pages[pages >= 0]
    assert np.array_equal(bits16(d["k_pool"][torch.from_numpy(pages).cuda()]), kp[pages])
    assert np.array_equal(bits16(d["v_pool"][torch.from_numpy(pages).cuda()]), vp[pages])


def _path(par, i):
    out = []
    while i >= 0:
        out.append(int(i))
        i = par[i]
    return out[::-1]


def test_commit_bad_page_flagged(cuda_dev):
    LT = _lt()
    cfg = W.VerifyConfig("commit-bad", ctx=(63,), Hq=2, Hkv=1, D=128, dtype=W.BF16, N=4, vocab=8,
                         paged="permuted", spare_pages=1)
    inp = W.generate(cfg, seed=4)
    inp["page_table"] = inp["page_table"].copy()
    inp["page_table"][0, 1] = -1
    acc = np.array([[0, 1, 2, 3]], np.int32)
    d, ctx_out, st = _gpu_commit(inp, cfg, acc, np.array([4], np.int32))
    assert st & LT.DEV_BAD_PAGE
    assert ctx_out.item() == 64  # stopped at the first position that has no page


# ---------------------------------------------------------------- the whole step

def test_full_step_matches_oracle(cuda_dev):
    import torch
    LT = _lt()
    cfg = W.GQA27B_32K
    inp = cached_inputs(cfg)
    d = to_device(inp, cfg)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    step.run(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
             d["parent"], d["draft"], d["logits"])
    torch.cuda.synchronize()
    am = oracle.argmax(inp["logits"])
    acc, alen, bonus = oracle.accept(inp["parent"], inp["draft"], am)
    assert step.status.item() == 0
    assert np.array_equal(step.argmax.cpu().numpy(), am)
    assert np.array_equal(step.acc_nodes.cpu().numpy(), acc)
    assert np.array_equal(step.acc_len.cpu().numpy(), alen)
    assert np.array_equal(step.bonus.cpu().numpy(), bonus)
    assert step.ctx_out.cpu().numpy()[0] == inp["ctx_len"][0] + alen[0]


@pytest.mark.slow
def test_argmax_and_accept_every_sweep_point_on_gpu(cuda_dev):
    """The sweep's 27 points: argmax on the GPU bit-exact against the oracle's
    linear scan, then acceptance from the GPU's own argmax."""
    import torch
    LT = _lt()
    for cfg in W.sweep_points():
        inp = W.generate(cfg, seed=5, with_pools=False)
        rows = cfg.B * (cfg.N + 1)
        xt = torch.from_numpy(inp["logits"]).cuda()
        out = torch.full((cfg.B, cfg.N + 1), -7, dtype=torch.int32, device="cuda")
        ws = torch.empty(LT.lucetree_argmax_workspace(rows, cfg.vocab), dtype=torch.uint8, device="cuda")
        LT.lucetree_argmax(xt, out, ws)
        am = oracle.argmax(inp["logits"])
        assert np.array_equal(out.cpu().numpy(), am), cfg.name
        acc, alen, bonus, st = _gpu_accept(inp["parent"], inp["draft"], out.cpu().numpy(), cfg.vocab)
        racc, ralen, rbonus = oracle.accept(inp["parent"], inp["draft"], am)
        assert st == 0
        assert np.array_equal(acc, racc) and np.array_equal(alen, ralen) and np.array_equal(bonus, rbonus), cfg.name


@pytest.mark.slow
def test_full_step_sweep_point_full_pool_compare(cuda_dev):
    """One whole step on the 4-sequence sweep pool (budget 40, random tree,
    planted match 0.95): argmax, acceptance and the commit are bit-exact, and
    every byte of both 1.6 GiB pools equals the oracle's commit."""
    import torch
    LT = _lt()
    cfg = [c for c in W.sweep_points() if c.N == 40 and c.tree == "random" and c.p_plant == 0.95][0]
    inp = W.generate(cfg, seed=11)
    d = to_device(inp, cfg)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    step.run(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
             d["parent"], d["draft"], d["logits"])
    torch.cuda.synchronize()
    am = oracle.argmax(inp["logits"])
    acc, alen, bonus = oracle.accept(inp["parent"], inp["draft"], am)
    assert alen.sum() > cfg.B  # the planting makes multi-node paths
    assert step.status.item() == 0
    assert np.array_equal(step.argmax.cpu().numpy(), am)
    assert np.array_equal(step.acc_nodes.cpu().numpy(), acc)
    assert np.array_equal(step.acc_len.cpu().numpy(), alen) and np.array_equal(step.bonus.cpu().numpy(), bonus)
    kp, vp, ctx = oracle.commit(inp, acc, alen, inplace=True)
    assert np.array_equal(step.ctx_out.cpu().numpy(), ctx)
    assert np.array_equal(bits16(d["k_pool"]), kp)
    assert np.array_equal(bits16(d["v_pool"]), vp)


# ---------------------------------------------------------------- the fused step (one C call)

def _inputs_step(cfg, seed):
    inp = W.generate(cfg, seed=seed)
    return inp, to_device(inp, cfg)


@pytest.mark.parametrize("name", ["ragged-f16-d128", "multi-bf16-d256"])
def test_fused_step_equals_the_five_calls(cuda_dev, name):
    """lucetree_verify_step gives bit for bit what the five separate calls
    give: attention output and lse, argmax, acceptance, and the pools and
    lengths after the commit."""
    import torch
    LT = _lt()
    if name == "ragged-f16-d128":
        cfg = W.VerifyConfig(name, ctx=(0, 63, 65, 1000, 2049), Hq=12, Hkv=3, D=128, dtype=W.F16, N=9,
                             tree="random", branch_cap=3, vocab=3000, p_plant=0.9, paged="permuted", spare_pages=5)
    else:
        cfg = W.VerifyConfig(name, ctx=(4000, 130, 9000), Hq=24, Hkv=4, D=256, dtype=W.BF16, N=22,
                             tree="random", branch_cap=4, vocab=5000, p_plant=0.9, paged="permuted", spare_pages=6)
    inp, d1 = _inputs_step(cfg, 41)
    d2 = to_device(inp, cfg)
    s1 = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    s2 = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    args = lambda d: (d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
                      d["parent"], d["draft"], d["logits"])
    s1.run(*args(d1))
    s2.run_calls(*args(d2))
    torch.cuda.synchronize()
    assert s1.status.item() == 0 and s2.status.item() == 0
    for name_ in ("out", "lse", "argmax", "acc_nodes", "acc_len", "bonus", "ctx_out"):
        a, b = getattr(s1, name_), getattr(s2, name_)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name_
    assert torch.equal(d1["k_pool"].view(torch.int16), d2["k_pool"].view(torch.int16))
    assert torch.equal(d1["v_pool"].view(torch.int16), d2["v_pool"].view(torch.int16))
    assert s1.acc_len.sum().item() > 0


def test_fused_step_repeated_calls_are_identical(cuda_dev):
    """Twenty fused steps on the same inputs (the commit rewrites the same
    rows each time) give bitwise identical results and a clean status: a
    race between the kernels' roles would show up as a difference."""
    import torch
    LT = _lt()
    cfg = W.VerifyConfig("repeat", ctx=(20000, 3000), Hq=24, Hkv=4, D=256, dtype=W.BF16, N=22, tree="random",
                         branch_cap=4, vocab=20000, p_plant=0.9, paged="permuted", spare_pages=4)
    inp, d = _inputs_step(cfg, 43)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    args = (d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"], d["parent"],
            d["draft"], d["logits"])
    step.run(*args)
    torch.cuda.synchronize()
    first = {k: getattr(step, k).clone() for k in ("out", "lse", "argmax", "acc_nodes", "acc_len", "bonus", "ctx_out")}
    for _ in range(19):
        step.run(*args)
    torch.cuda.synchronize()
    assert step.status.item() == 0
    for k, v in first.items():
        assert torch.equal(getattr(step, k).view(torch.int32), v.view(torch.int32)), k
    ref, _ = oracle.verify_attn(inp, oracle.BF16)
    from tests.helpers import ATTN_TOL, row_error
    assert row_error(step.out.cpu().numpy().reshape(-1, cfg.D), ref).max() <= ATTN_TOL


def test_fused_step_host_and_device_checks(cuda_dev):
    import torch
    LT = _lt()
    cfg = W.VerifyConfig("step-bad", ctx=(300, 100), Hq=4, Hkv=2, D=128, dtype=W.F16, N=5, vocab=50,
                         paged="permuted", spare_pages=2)
    inp, d = _inputs_step(cfg, 44)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    # the new lengths may not overwrite the old ones: merge CTAs still read them
    with pytest.raises(LT.LucetreeError):
        LT._step_args(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
                      d["parent"], d["draft"], d["logits"], step.out, step.lse, step.argmax, step.acc_nodes,
                      step.acc_len, step.bonus, d["ctx_len"], step.status)
    s = LT._step_args(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
                      d["parent"], d["draft"], d["logits"], step.out, step.lse, step.argmax, step.acc_nodes,
                      step.acc_len, step.bonus, step.ctx_out, step.status)
    lib = LT.load()
    import ctypes
    s.ctx_len_out = s.attn.ctx_len
    assert lib.lucetree_verify_step(ctypes.byref(s), LT._ptr(step.ws_step), step.ws_step.numel(), None) == 1
    s.ctx_len_out = LT._ptr(step.ctx_out)
    assert lib.lucetree_verify_step(ctypes.byref(s), LT._ptr(step.ws_step), 16, None) == 3  # workspace too small
    # a parent that is not an earlier node is flagged on the device, the call completes
    bad = d["parent"].clone()
    bad[1, 3] = 4
    step.run(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"], bad,
             d["draft"], d["logits"])
    torch.cuda.synchronize()
    assert step.status.item() & LT.DEV_BAD_PARENT
    assert step.acc_len[1].item() == 0
