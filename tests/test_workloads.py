"""Structure of the seeded synthetic workloads (CPU)."""
import numpy as np

import workloads as W


def test_random_tree_respects_cap_and_order():
    rng = np.random.default_rng(0)
    for n in (1, 8, 22, 40, 64):
        par = W.random_parents(rng, n, "random", 4)
        assert par[0] == -1
        assert all(-1 <= par[i] < i for i in range(n))
        assert all(p >= 0 for p in par[1:])
        counts = np.bincount(par[1:], minlength=n) if n > 1 else np.zeros(1)
        assert counts.max() <= 4


def test_chain_tree():
    par = W.random_parents(np.random.default_rng(0), 9, "chain", 4)
    assert list(par) == [-1] + list(range(8))


def test_sibling_drafts_distinct():
    rng = np.random.default_rng(1)
    par = W.random_parents(rng, 64, "random", 4)
    dr = W.draft_tokens(rng, par, 5)
    for p in set(par.tolist()):
        toks = dr[par == p]
        assert len(set(toks.tolist())) == len(toks)


def test_planting_rate():
    rng = np.random.default_rng(2)
    hits = total = 0
    for _ in range(400):
        par = W.random_parents(rng, 8, "random", None)
        dr = W.draft_tokens(rng, par, 4096)
        lg = W.planted_logits(rng, par, dr, 4096, 0.7)
        am = np.argmax(lg, axis=1)
        for p in set(par.tolist()):
            total += 1
            hits += any(dr[c] == am[p + 1] for c in np.nonzero(par == p)[0])
    assert abs(hits / total - 0.7) < 0.05


def test_paged_layout_and_determinism():
    cfg = W.TINY.replace(ctx=(100, 0, 640), N=5, D=8, paged="permuted", spare_pages=7)
    a = W.generate(cfg, seed=4)
    b = W.generate(cfg, seed=4)
    for k in a:
        assert np.array_equal(a[k], b[k])
    pt = a["page_table"]
    used = pt[pt >= 0]
    assert len(np.unique(used)) == len(used)
    assert a["k_pool"].shape[0] == len(used) + 7
    for bi, L in enumerate(cfg.ctx):
        assert (pt[bi] >= 0).sum() == W.pages_needed(L, cfg.N)
    # committed slots are finite, everything else is NaN
    k = a["k_pool"]
    nan = W.NAN_BITS[W.F16]
    assert (k[pt[0, 0]] != nan).all()
    assert (k[pt[0, 1], :, :36] != nan).all() and (k[pt[0, 1], :, 36:] == nan).all()
    assert (k[pt[1, 0]] == nan).all()


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    bits = W.f32_to_bf16_bits(x)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    assert back[0] == 1.0
    assert back[1] == 1.0                      # tie -> even
    assert back[2] == 1.0 + 2 ** -6            # tie -> even (up)
    assert back[3] == -2.5


def test_sweep_has_27_points():
    pts = W.sweep_points()
    assert len(pts) == 27
    assert len({p.name for p in pts}) == 27
