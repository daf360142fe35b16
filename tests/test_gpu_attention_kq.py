"""Tree-verify attention with K stored as FP8 E4M3 codes (one power-of-two
exponent per token and head) through the C-ABI, against the fp64 oracle run
on the exactly dequantised K (and V, where V is quantised too).  Same 2e-3
row bar as the 16-bit path: the queries' two-part E4M3 split reproduces bf16
queries to far below it.  Also the commit into an E4M3 K pool, byte-exact
against the oracle's commit_kq, and a second step over the committed pool."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import ATTN_TOL, bits16, row_error, to_device

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _run_kq(cfg, inp, kq, v_format=0, vq=None, lse=False):
    import torch
    LT = _lt()
    d = to_device(inp, cfg)
    B, N, Hq, Hkv, D = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D
    anc = torch.empty(B, N, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_build_anc_mask(d["parent"], anc, st)
    ws = torch.empty(LT.lucetree_verify_attn_kq_workspace(B, N, Hq, Hkv, D), dtype=torch.uint8, device="cuda")
    ws.fill_(0x3F)
    out = torch.full((B, N, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse_t = torch.full((B, N, Hq), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    kc = torch.from_numpy(kq["k_codes"]).cuda()
    ke = torch.from_numpy(kq["k_exp"]).cuda()
    if v_format:
        vpool = torch.from_numpy(vq["v_codes"]).cuda()
        vexp = torch.from_numpy(vq["v_exp"]).cuda()
    else:
        vpool, vexp = d["v_pool"], None
    LT.lucetree_verify_attn_kq(d["q"], kc, ke, vpool, d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"], anc,
                               out, st, ws, v_format=v_format, v_exp=vexp, lse=lse_t)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(-1, D), (lse_t.cpu().numpy().reshape(-1) if lse else None), st.item()


def _reference(cfg, inp, kq, v_format=0, vq=None):
    ref = dict(inp)
    ref["k_pool"] = oracle.dequant_k_e4m3(kq["k_codes"], kq["k_exp"], oracle.BF16)
    if v_format:
        ref["v_pool"] = oracle.dequant_v(vq["v_codes"], vq["v_exp"], v_format, oracle.BF16)
    return oracle.verify_attn(ref, oracle.BF16)


def _check(cfg, seed, v_format=0, lse=True, dist="normal"):
    inp = W.generate(cfg, seed=seed, with_logits=False)
    kq = W.generate_kq(cfg, seed=seed, dist=dist)
    vq = W.generate_vq(cfg, v_format, seed=seed) if v_format else None
    got, got_lse, status = _run_kq(cfg, inp, kq, v_format, vq, lse=lse)
    assert status == 0
    ref, ref_lse = _reference(cfg, inp, kq, v_format, vq)
    assert np.isfinite(got).all()
    err = row_error(got, ref.reshape(got.shape))
    assert err.max() <= ATTN_TOL, f"worst row {err.argmax()}: {err.max():.3e}"
    if lse:
        assert np.abs(got_lse - ref_lse).max() <= 1e-3 * np.maximum(1.0, np.abs(ref_lse)).max()


@pytest.mark.parametrize("dist", ["normal", "uniform"])
@pytest.mark.parametrize("v_format", [0, W.V_INT8, W.V_INT4], ids=["bf16v", "int8v", "int4v"])
def test_kq_ragged_batch(cuda_dev, v_format, dist):
    # committed lengths straddle tile (128) and page (64) boundaries, one is empty; codes spread over the
    # whole E4M3 range ("uniform") move the running maxima on most tiles
    cfg = W.VerifyConfig("kq-ragged", ctx=(0, 1, 63, 65, 127, 129, 1000, 2049), Hq=12, Hkv=3, D=256, dtype=W.BF16,
                         N=9, tree="random", branch_cap=3, vocab=512, paged="permuted", spare_pages=5)
    _check(cfg, 21, v_format, dist=dist)


@pytest.mark.parametrize("v_format", [0, W.V_INT8], ids=["bf16v", "int8v"])
def test_kq_several_segments_per_cta_budget_22(cuda_dev, v_format):
    cfg = W.VerifyConfig("kq-multiseg", ctx=(4000, 3000, 2000, 4100, 130, 5000, 64, 3333), Hq=24, Hkv=4, D=256,
                         dtype=W.BF16, N=22, tree="random", branch_cap=4, vocab=512, paged="permuted", spare_pages=4)
    _check(cfg, 32, v_format)


@pytest.mark.parametrize("N,shape", [(1, "chain"), (40, "random"), (64, "chain")])
def test_kq_budgets_cover_row_groups(cuda_dev, N, shape):
    cfg = W.VerifyConfig(f"kq-budget{N}", ctx=(3000, 700), Hq=24, Hkv=4, D=256, dtype=W.BF16, N=N, tree=shape,
                         branch_cap=4, vocab=256, paged="permuted", spare_pages=3)
    _check(cfg, N, 0)


@pytest.mark.slow
@pytest.mark.parametrize("v_format", [0, W.V_INT8], ids=["bf16v", "int8v"])
def test_kq_headline_128k_all_rows(cuda_dev, v_format):
    _check(W.HEADLINE_128K_B22, 0, v_format)


def test_kq_zero_exponents_read_as_zero(cuda_dev):
    cfg = W.VerifyConfig("kq-zero", ctx=(700,), Hq=6, Hkv=1, D=256, dtype=W.BF16, N=4, vocab=64)
    inp = W.generate(cfg, seed=3, with_logits=False)
    kq = W.generate_kq(cfg, seed=3)
    kq["k_exp"][:] = 0
    got, _, status = _run_kq(cfg, inp, kq)
    ref, _ = _reference(cfg, inp, kq)
    assert status == 0 and row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL


def test_kq_refuses_fp16_and_head_dim_128(cuda_dev):
    LT = _lt()
    for dtype, D in ((W.F16, 256), (W.BF16, 128)):
        cfg = W.VerifyConfig("kq-bad", ctx=(100,), Hq=4, Hkv=1, D=D, dtype=dtype, N=2, vocab=64)
        inp = W.generate(cfg, seed=1, with_logits=False)
        kq = W.generate_kq(cfg, seed=1)
        with pytest.raises(LT.LucetreeError):
            _run_kq(cfg, inp, kq)


def test_commit_kq_byte_exact_then_second_step(cuda_dev):
    """Commit the accepted path into the E4M3 K pool (and the bf16 V pool):
    codes, exponents, V and lengths equal the oracle's commit byte for byte;
    a second verify step over the committed pool matches the oracle."""
    import torch
    LT = _lt()
    cfg = W.VerifyConfig("kq-commit", ctx=(190, 64, 1000), Hq=8, Hkv=2, D=256, dtype=W.BF16, N=10, tree="random",
                         branch_cap=3, vocab=300, p_plant=0.95, paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=13)
    kq = W.generate_kq(cfg, seed=13)
    am = oracle.argmax(inp["logits"])
    acc, alen, _ = oracle.accept(inp["parent"], inp["draft"], am)
    assert alen.sum() > cfg.B
    ref_codes, ref_exp = oracle.commit_kq(dict(inp, dtype_id=oracle.BF16), kq["k_codes"], kq["k_exp"], acc, alen)
    _, ref_v, ref_ctx = oracle.commit(inp, acc, alen)
    d = to_device(inp, cfg)
    kc = torch.from_numpy(kq["k_codes"]).cuda()
    ke = torch.from_numpy(kq["k_exp"]).cuda()
    ctx_out = torch.empty_like(d["ctx_len"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_commit_kq(d["k_tree"], d["v_tree"], torch.from_numpy(acc).cuda(), torch.from_numpy(alen).cuda(),
                          d["page_table"], d["ctx_len"], ctx_out, kc, ke, d["v_pool"], st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(kc.cpu().numpy(), ref_codes) and np.array_equal(ke.cpu().numpy(), ref_exp)
    assert np.array_equal(bits16(d["v_pool"]), ref_v) and np.array_equal(ctx_out.cpu().numpy(), ref_ctx)
    # the next step attends over the committed (quantised) prefix
    nxt = W.generate(cfg, seed=14, with_logits=False)
    inp2 = dict(inp, v_pool=ref_v, ctx_len=ref_ctx, q=nxt["q"], k_tree=nxt["k_tree"], v_tree=nxt["v_tree"],
                parent=nxt["parent"])
    got, _, status = _run_kq(cfg, inp2, dict(k_codes=ref_codes, k_exp=ref_exp))
    ref, _ = _reference(cfg, inp2, dict(k_codes=ref_codes, k_exp=ref_exp))
    assert status == 0 and row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL
