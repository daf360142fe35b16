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


def _f64(bits, dtype):
    bits = np.asarray(bits, np.uint16)
    if dtype == W.BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def test_delta_inputs_follow_their_recipe():
    cfg = W.DeltaConfig("gen-delta", B=3, N=22, Hk=2, Hv=4, dk=128, dv=64, dtype=W.BF16, tree="random", branch_cap=4)
    a = W.generate_delta(cfg, seed=1)
    assert a["q"].shape == a["k"].shape == (3, 22, 2, 128) and a["q"].dtype == np.uint16
    assert a["v"].shape == (3, 22, 4, 64) and a["state"].shape == (3, 4, 128, 64)
    assert a["alpha"].dtype == a["beta"].dtype == a["state"].dtype == np.float32
    for key in ("q", "k"):  # unit vectors up to the dtype's rounding
        n = np.linalg.norm(_f64(a[key], cfg.dtype), axis=-1)
        assert np.abs(n - 1.0).max() < 2 ** -7
    # alpha = exp(-0.1 softplus(z)) lies in (0, 1); beta = sigmoid(z) in (0, 1)
    assert (a["alpha"] > 0).all() and (a["alpha"] < 1).all() and (a["beta"] > 0).all() and (a["beta"] < 1).all()
    assert np.exp(-0.1 * np.log1p(np.exp(5.0))) < a["alpha"].min() and abs(float(a["beta"].mean()) - 0.5) < 0.05
    assert abs(float(a["state"].std()) - 0.1) < 0.005
    for b in range(3):
        par = a["parent"][b]
        assert par[0] == -1 and all(-1 <= par[i] < i for i in range(22))
        assert np.bincount(par[par >= 0], minlength=22).max() <= 4
    b = W.generate_delta(cfg, seed=1)
    c = W.generate_delta(cfg, seed=2)
    assert all(np.array_equal(a[k], b[k]) for k in a) and not np.array_equal(a["v"], c["v"])


def test_quantised_storage_inputs_follow_their_recipe():
    cfg = W.VerifyConfig("gen-vq", ctx=(700, 64), Hq=6, Hkv=3, D=256, dtype=W.BF16, N=5, paged="permuted",
                         spare_pages=2)
    pools = W.generate(cfg, seed=0)["k_pool"].shape
    v8 = W.generate_vq(cfg, W.V_INT8, seed=0)
    assert v8["v_codes"].shape == pools and v8["v_codes"].dtype == np.uint8
    c8 = v8["v_codes"].view(np.int8)
    assert c8.min() >= -127 and c8.max() <= 127 and c8.min() < -100 and c8.max() > 100
    assert v8["v_exp"].shape == pools[:3] and v8["v_exp"].min() >= 118 and v8["v_exp"].max() <= 124
    v4 = W.generate_vq(cfg, W.V_INT4, seed=0)
    assert v4["v_codes"].shape == pools[:3] + (cfg.D // 2,)
    nib = np.stack([v4["v_codes"] & 0xF, v4["v_codes"] >> 4]).astype(np.int64)
    signed = np.where(nib >= 8, nib - 16, nib)
    assert signed.min() == -7 and signed.max() == 7  # the code -8 is never drawn
    kq = W.generate_kq(cfg, seed=0, dist="uniform")
    assert kq["k_codes"].shape == pools and not ((kq["k_codes"] & 0x7F) == 0x7F).any()  # no NaN codes
    assert kq["k_exp"].min() >= 120 and kq["k_exp"].max() <= 124
    assert len(np.unique(kq["k_codes"])) == 254
    import oracle
    kn = W.generate_kq(cfg, seed=0)  # the "normal" draw: N(0, 160^2) values toward zero
    assert kn["k_codes"].shape == pools and not ((kn["k_codes"] & 0x7F) == 0x7F).any()
    v = oracle.decode_e4m3(kn["k_codes"])
    assert abs(v.std() - 160.0) < 8.0 and np.abs(v).max() == 448.0
    assert kn["k_exp"].min() == 119 and kn["k_exp"].max() == 120


def test_lmhead_inputs_follow_their_recipe():
    cfg = W.LmHeadConfig("gen-lm", rows=9, d_model=256, vocab=5000, dtype=W.F16)
    a = W.generate_lmhead(cfg, seed=0)
    assert a["hidden"].shape == (9, 256) and a["weight"].shape == (5000, 256)
    assert a["hidden"].dtype == a["weight"].dtype == np.uint16
    assert abs(float(_f64(a["hidden"], cfg.dtype).std()) - 1.0) < 0.05
    assert abs(float(_f64(a["weight"], cfg.dtype).std()) - cfg.w_std) < 0.001


def test_e4m3_code_toward_zero_bit_construction():
    """The generator's code draw: the code's value never exceeds |x| and the
    next larger code does (values below 448), signs follow x, no NaN codes."""
    import oracle
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(50000) * 160.0, rng.standard_normal(5000) * 1e-3, [0.0, -0.0, 448.0,
                                                                                                 -600.0, 2.0 ** -9]])
    c = W.e4m3_code_toward_zero(x)
    assert not ((c & 0x7F) == 0x7F).any()
    v = oracle.decode_e4m3(c)
    a = np.minimum(np.abs(x), 448.0)
    assert (np.abs(v) <= a).all()
    vals = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    up = vals[np.minimum(np.searchsorted(vals, np.abs(v)) + 1, len(vals) - 1)]
    assert ((up > a) | (np.abs(v) == 448.0)).all()
    assert (np.signbit(v) == np.signbit(x)).all()
    assert W.e4m3_code_toward_zero(np.array([1.0, 448.0, 2.0 ** -9])).tolist() == [0x38, 0x7E, 0x01]
