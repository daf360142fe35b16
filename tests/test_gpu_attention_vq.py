"""Tree-verify attention with V stored quantised (int8 / int4 codes with one
power-of-two exponent per token and head) through the C-ABI, against the fp64
oracle run on the exactly dequantised V.  Same 2e-3 row bar as the 16-bit
path: dequantisation into the on-chip fp16 operand is exact."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import ATTN_TOL, oracle_dtype, row_error, to_device

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _run_vq(cfg, inp, vq, v_format, rows=None):
    import torch
    LT = _lt()
    d = to_device(inp, cfg)
    B, N, Hq, Hkv, D = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D
    anc = torch.empty(B, N, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_build_anc_mask(d["parent"], anc, st)
    ws = torch.empty(LT.lucetree_verify_attn_workspace(B, N, Hq, Hkv, D), dtype=torch.uint8, device="cuda")
    out = torch.full((B, N, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    codes = torch.from_numpy(vq["v_codes"]).cuda()
    vexp = torch.from_numpy(vq["v_exp"]).cuda()
    LT.lucetree_verify_attn_vq(d["q"], d["k_pool"], codes, vexp, v_format, d["page_table"], d["ctx_len"],
                               d["k_tree"], d["v_tree"], anc, out, st, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(-1, D), st.item()


def _reference(cfg, inp, vq, v_format, rows=None):
    ref_inp = dict(inp)
    ref_inp["v_pool"] = oracle.dequant_v(vq["v_codes"], vq["v_exp"], v_format, oracle_dtype(cfg))
    return oracle.verify_attn(ref_inp, oracle_dtype(cfg), rows=rows)[0]


@pytest.mark.parametrize("v_format", [W.V_INT8, W.V_INT4], ids=["int8", "int4"])
@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
def test_quantised_v_ragged_batch(cuda_dev, dtype, v_format):
    cfg = W.VerifyConfig("vq-ragged", ctx=(0, 1, 63, 65, 127, 129, 1000, 2049), Hq=12, Hkv=3, D=256, dtype=dtype,
                         N=9, tree="random", branch_cap=3, vocab=512, paged="permuted", spare_pages=5)
    inp = W.generate(cfg, seed=21)
    vq = W.generate_vq(cfg, v_format, seed=21)
    got, status = _run_vq(cfg, inp, vq, v_format)
    assert status == 0
    ref = _reference(cfg, inp, vq, v_format)
    err = row_error(got, ref.reshape(got.shape))
    assert err.max() <= ATTN_TOL, err.max()


@pytest.mark.parametrize("v_format", [W.V_INT8, W.V_INT4], ids=["int8", "int4"])
def test_quantised_v_budgets_and_segments(cuda_dev, v_format):
    # several key segments per CTA, and the 144-row group of budget 22
    cfg = W.VerifyConfig("vq-multiseg", ctx=(4000, 3000, 2000, 4100, 130, 5000, 64, 3333), Hq=24, Hkv=4, D=256,
                         dtype=W.BF16, N=22, tree="random", branch_cap=4, vocab=512, paged="permuted", spare_pages=4)
    inp = W.generate(cfg, seed=32)
    vq = W.generate_vq(cfg, v_format, seed=32)
    got, status = _run_vq(cfg, inp, vq, v_format)
    assert status == 0
    ref = _reference(cfg, inp, vq, v_format)
    assert row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL


@pytest.mark.slow
@pytest.mark.parametrize("v_format", [W.V_INT8, W.V_INT4], ids=["int8", "int4"])
def test_quantised_v_headline_128k_all_rows(cuda_dev, v_format):
    cfg = W.HEADLINE_128K_B22
    inp = W.generate(cfg, seed=0, with_logits=False)
    vq = W.generate_vq(cfg, v_format, seed=0)
    got, status = _run_vq(cfg, inp, vq, v_format)
    assert status == 0
    ref = _reference(cfg, inp, vq, v_format)
    assert row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL


def test_quantised_v_zero_exponents_read_as_zero(cuda_dev):
    cfg = W.VerifyConfig("vq-zero", ctx=(700,), Hq=6, Hkv=1, D=256, dtype=W.BF16, N=4, vocab=64)
    inp = W.generate(cfg, seed=3)
    vq = W.generate_vq(cfg, W.V_INT8, seed=3)
    vq["v_exp"][:] = 0
    got, status = _run_vq(cfg, inp, vq, W.V_INT8)
    zero = dict(inp)
    zero["v_pool"] = np.zeros_like(inp["v_pool"])
    ref = oracle.verify_attn(zero, oracle_dtype(cfg))[0]
    assert status == 0 and row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL


@pytest.mark.parametrize("v_format", [W.V_INT8, W.V_INT4], ids=["int8", "int4"])
def test_quantised_v_exponents_across_fp16_range(cuda_dev, v_format):
    # per-token exponents from 2^-31 to 2^9 (every code times its power of two stays an fp16
    # number or underflows to an fp16 subnormal), some zero: rows whose scale and 1152 (1032)
    # times it are fp16 numbers and rows whose are not expand by different routes on chip
    cfg = W.VerifyConfig("vq-exprange", ctx=(3000, 130, 1025), Hq=12, Hkv=3, D=256, dtype=W.BF16, N=9,
                         tree="random", branch_cap=3, vocab=512, paged="permuted", spare_pages=3)
    inp = W.generate(cfg, seed=41)
    vq = W.generate_vq(cfg, v_format, seed=41)
    rng = np.random.default_rng(41)
    e = rng.integers(96, 137, size=vq["v_exp"].shape)
    e[rng.random(e.shape) < 0.05] = 0
    vq["v_exp"][:] = e.astype(np.uint8)
    got, status = _run_vq(cfg, inp, vq, v_format)
    assert status == 0
    ref = _reference(cfg, inp, vq, v_format)
    assert row_error(got, ref.reshape(got.shape)).max() <= ATTN_TOL


def test_quantised_v_refuses_head_dim_128(cuda_dev):
    import torch
    LT = _lt()
    cfg = W.VerifyConfig("vq-d128", ctx=(100,), Hq=4, Hkv=1, D=128, dtype=W.BF16, N=2, vocab=64)
    inp = W.generate(cfg, seed=1)
    vq = W.generate_vq(cfg, W.V_INT8, seed=1)
    with pytest.raises(LT.LucetreeError):
        _run_vq(cfg, inp, vq, W.V_INT8)
