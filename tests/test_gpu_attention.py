"""Tree-verify attention through the C-ABI against the fp64 oracle.

Bar: for every compared row, max_d |gpu - oracle| / max_d |oracle| <= 2e-3
(bf16 / fp16 inputs, fp32 accumulation; the tolerance the workload states).
Every output row is compared, at every size, including the five workloads'
full sizes and every (budget, tree shape) pair of the concurrent sweep.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import ATTN_TOL, bits16, cached_inputs, oracle_dtype, row_error, run_attention, to_device

pytestmark = pytest.mark.gpu


def _check(cfg, inp, rows=None, lse=True, seed_rows=1):
    d = to_device(inp, cfg)
    out, lse_t, status = run_attention(d, cfg, lse=lse)
    assert status == 0
    out = out.cpu().numpy().reshape(-1, cfg.D)
    if rows is None:
        rows = np.arange(out.shape[0], dtype=np.int32)
    ref, ref_lse = oracle.verify_attn(inp, oracle_dtype(cfg), rows=rows)
    got = out[rows]
    assert np.isfinite(got).all()
    err = row_error(got, ref)
    assert err.max() <= ATTN_TOL, f"worst row {rows[err.argmax()]}: {err.max():.3e}"
    if lse:
        gl = lse_t.cpu().numpy().reshape(-1)[rows]
        assert np.abs(gl - ref_lse).max() <= 1e-3 * np.maximum(1.0, np.abs(ref_lse)).max()
    return err


def test_tiny_all_rows(cuda_dev):
    cfg = W.TINY
    _check(cfg, cached_inputs(cfg))


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("D", [128, 256])
def test_small_ragged_batch_both_dtypes(cuda_dev, dtype, D):
    # committed lengths straddle tile (128) and page (64) boundaries, one is empty
    cfg = W.VerifyConfig("ragged", ctx=(0, 1, 63, 65, 127, 129, 1000, 2049), Hq=12, Hkv=3, D=D, dtype=dtype,
                         N=9, tree="random", branch_cap=3, vocab=512, paged="permuted", spare_pages=5)
    _check(cfg, W.generate(cfg, seed=21))


@pytest.mark.parametrize("dtype", [W.F16, W.BF16])
@pytest.mark.parametrize("D", [128, 256])
def test_several_key_segments_per_cta(cuda_dev, dtype, D):
    # 700 tiles over the SMs: most CTAs cross key-segment boundaries, so a
    # segment's epilogue runs while the next segment's K/V are already landing
    cfg = W.VerifyConfig("multiseg", ctx=(4000, 3000, 2000, 4100, 130, 5000, 64, 3333), Hq=16, Hkv=4, D=D,
                         dtype=dtype, N=9, tree="random", branch_cap=3, vocab=512, paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=31)
    _check(cfg, inp)


def test_bf16_v_beyond_fp16_range_is_flagged_nonfinite(cuda_dev):
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    cfg = W.VerifyConfig("vrange", ctx=(300,), Hq=4, Hkv=2, D=128, dtype=W.BF16, N=3, vocab=64)
    inp = W.generate(cfg, seed=8)
    d = to_device(inp, cfg)
    _, _, status = run_attention(d, cfg)
    assert status == 0
    page = int(inp["page_table"][0, 2])  # committed position 130 of sequence 0
    d["v_pool"][page, 1, 2, 5] = 1.0e5
    _, _, status = run_attention(d, cfg)
    assert status & LT.DEV_NONFINITE


@pytest.mark.parametrize("N,shape", [(1, "chain"), (8, "chain"), (22, "random"), (40, "random"), (64, "random"),
                                     (64, "chain")])
def test_budgets_cover_row_groups(cuda_dev, N, shape):
    # 24 query heads over 4 KV heads: N*6 rows split into 1..3 row groups
    cfg = W.VerifyConfig(f"budget{N}", ctx=(3000, 700), Hq=24, Hkv=4, D=256, dtype=W.BF16, N=N, tree=shape,
                         branch_cap=4, vocab=256, paged="permuted", spare_pages=3)
    _check(cfg, W.generate(cfg, seed=N))


def test_gqa27b_32k_all_rows(cuda_dev):
    cfg = W.GQA27B_32K
    _check(cfg, cached_inputs(cfg))


@pytest.mark.slow
def test_long_128k_b40_all_rows(cuda_dev):
    cfg = W.LONG_128K
    _check(cfg, cached_inputs(cfg))


@pytest.mark.slow
def test_headline_128k_b22_all_rows(cuda_dev):
    # the workload bench.py times: one sequence, 131072 committed tokens on
    # permuted pages, budget 22 (one row group of 132 rows per KV head)
    cfg = W.HEADLINE_128K_B22
    _check(cfg, cached_inputs(cfg))


@pytest.mark.slow
def test_paged_256k_all_rows(cuda_dev):
    cfg = W.PAGED_256K
    _check(cfg, cached_inputs(cfg))


SWEEP_SHAPES = [(1, "chain"), (8, "chain"), (8, "random"), (22, "chain"), (22, "random"), (40, "chain"),
                (40, "random"), (64, "chain"), (64, "random")]


@pytest.mark.slow
@pytest.mark.parametrize("N,shape", SWEEP_SHAPES)
def test_concurrent_sweep_point_all_rows(cuda_dev, N, shape):
    # four ragged sequences {4K, 32K, 128K, 256K} in one permuted pool; the
    # attention rows do not depend on the planting probability (logits only)
    cfg = [c for c in W.sweep_points() if c.N == N and c.tree == shape and c.p_plant == 0.7][0]
    _check(cfg, W.generate(cfg, seed=3, with_logits=False), lse=N in (1, 64))


def test_non_ancestor_tree_kv_is_invisible(cuda_dev):
    cfg = W.VerifyConfig("mask", ctx=(500,), Hq=8, Hkv=2, D=128, dtype=W.BF16, N=16, tree="random",
                         vocab=64)
    inp = W.generate(cfg, seed=5)
    anc = oracle.ancestor_matrix(inp["parent"][0])
    i = 15
    non = [j for j in range(cfg.N) if not anc[i, j]]
    assert non
    base, _, _ = run_attention(to_device(inp, cfg), cfg)
    pert = dict(inp)
    rng = np.random.default_rng(0)
    pert["k_tree"] = inp["k_tree"].copy()
    pert["v_tree"] = inp["v_tree"].copy()
    pert["k_tree"][0, non] = W.f32_to_bf16_bits(rng.standard_normal(pert["k_tree"][0, non].shape) * 5)
    pert["v_tree"][0, non] = W.f32_to_bf16_bits(rng.standard_normal(pert["v_tree"][0, non].shape) * 5)
    out, _, _ = run_attention(to_device(pert, cfg), cfg)
    assert np.array_equal(out[0, i].cpu().numpy(), base[0, i].cpu().numpy())


def test_page_relabelling(cuda_dev):
    cfg = W.VerifyConfig("relabel", ctx=(900, 257), Hq=8, Hkv=2, D=256, dtype=W.BF16, N=6, vocab=64,
                         paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=6)
    base, _, _ = run_attention(to_device(inp, cfg), cfg)
    perm = np.random.default_rng(2).permutation(inp["k_pool"].shape[0])
    moved = dict(inp)
    moved["k_pool"] = np.empty_like(inp["k_pool"])
    moved["v_pool"] = np.empty_like(inp["v_pool"])
    moved["k_pool"][perm] = inp["k_pool"]
    moved["v_pool"][perm] = inp["v_pool"]
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    moved["page_table"] = pt
    out, _, _ = run_attention(to_device(moved, cfg), cfg)
    err = row_error(out.cpu().numpy().reshape(-1, cfg.D), base.cpu().numpy().reshape(-1, cfg.D).astype(np.float64))
    assert err.max() <= ATTN_TOL


def test_bad_page_and_ctx_are_flagged(cuda_dev):
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    cfg = W.VerifyConfig("bad", ctx=(300, 200), Hq=4, Hkv=2, D=128, dtype=W.F16, N=3, vocab=64,
                         paged="permuted", spare_pages=2)
    inp = W.generate(cfg, seed=7)
    bad = dict(inp)
    bad["page_table"] = inp["page_table"].copy()
    bad["page_table"][0, 1] = 10_000
    _, _, status = run_attention(to_device(bad, cfg), cfg)
    assert status & LT.DEV_BAD_PAGE
    bad = dict(inp)
    bad["ctx_len"] = np.array([300, 10_000], np.int32)
    _, _, status = run_attention(to_device(bad, cfg), cfg)
    assert status & LT.DEV_BAD_CTX


def test_second_step_over_committed_cache(cuda_dev):
    """Step 1 commits its accepted path; step 2 attends over the longer prefix.
    The GPU's step 2 matches the oracle's step 2 run on the oracle's own commit."""
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    cfg = W.VerifyConfig("two-step", ctx=(190, 64), Hq=8, Hkv=2, D=128, dtype=W.BF16, N=10, tree="random",
                         branch_cap=3, vocab=300, p_plant=0.95, paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=13)
    am = oracle.argmax(inp["logits"])
    acc, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    assert alen.max() > 0
    kp, vp, ctx = oracle.commit(inp, acc, alen)
    d = to_device(inp, cfg)
    step = LT.VerifyStep(cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D, cfg.vocab)
    step.run(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"],
             d["parent"], d["draft"], d["logits"])
    torch.cuda.synchronize()
    assert np.array_equal(step.ctx_out.cpu().numpy(), ctx)
    # second step: fresh tree on top of the committed prefix
    nxt = W.generate(cfg, seed=14)
    inp2 = dict(inp, k_pool=kp, v_pool=vp, ctx_len=ctx, q=nxt["q"], k_tree=nxt["k_tree"], v_tree=nxt["v_tree"],
                parent=nxt["parent"])
    ref, _ = oracle.verify_attn(inp2, oracle_dtype(cfg))
    d2 = dict(d, ctx_len=step.ctx_out.clone(), q=to_device(nxt, cfg)["q"], k_tree=to_device(nxt, cfg)["k_tree"],
              v_tree=to_device(nxt, cfg)["v_tree"], parent=to_device(nxt, cfg)["parent"])
    out, _, status = run_attention(d2, cfg)
    assert status == 0
    assert row_error(out.cpu().numpy().reshape(-1, cfg.D), ref).max() <= ATTN_TOL
