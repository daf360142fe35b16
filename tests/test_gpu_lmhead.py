"""Fused lm_head projection + argmax through the C-ABI against the fp64 oracle.

The kernel multiplies 16-bit operands exactly and sums the products in fp32 on
the tensor cores; the oracle sums them in fp64.  The fp32 sum of n products
deviates from the exact one by rounding errors of at most 2^-24 of each
partial sum; modelled as independent, their total stays within
    tol = 8 * sqrt(n) * 2^-24 * sum_i |h_i w_i|
(the bound is per vocabulary row).  A row's pick j is therefore accepted when
its exact logit is within tol_j + tol_o of the oracle's maximum (o = the
oracle's pick); where the oracle's top two logits are further apart than
that, this forces j == o.  The returned logit is the kernel's fp32 value for
j, within tol_j of the exact one.  Exact ties (identical weight rows) must go
to the lowest index, bit-exact.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == W.BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return bits.view(np.float16).astype(np.float64)


def _odt(dtype: str) -> int:
    return oracle.BF16 if dtype == W.BF16 else oracle.F16


def _gpu(hidden: np.ndarray, weight: np.ndarray, dtype: str, reuse_ws=None):
    import torch
    LT = _lt()
    tdt = torch.bfloat16 if dtype == W.BF16 else torch.float16
    h = torch.from_numpy(np.ascontiguousarray(hidden).view(np.int16)).view(tdt).cuda()
    w = torch.from_numpy(np.ascontiguousarray(weight).view(np.int16)).view(tdt).cuda()
    rows = hidden.shape[0]
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    lg = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = reuse_ws
    if ws is None:
        ws = torch.empty(LT.lucetree_lmhead_argmax_workspace(rows), dtype=torch.uint8, device="cuda")
    LT.lucetree_lmhead_argmax(h, w, out, st, ws, out_logit=lg)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lg.cpu().numpy(), st.item(), ws


def _tol(h: np.ndarray, w_row: np.ndarray) -> float:
    return 8.0 * math.sqrt(h.shape[0]) * 2.0 ** -24 * float(np.abs(h) @ np.abs(w_row))


def _check(hidden, weight, dtype, idx, logit, min_exact=0.9):
    o_idx, top1, top2 = oracle.lmhead_argmax(hidden, weight, _odt(dtype))
    rows, vocab = hidden.shape[0], weight.shape[0]
    hf = _f64(hidden, dtype)
    assert np.all((idx >= 0) & (idx < vocab)), idx
    exact = 0
    for r in range(rows):
        j, o = int(idx[r]), int(o_idx[r])
        wj, wo = _f64(weight[j], dtype), _f64(weight[o], dtype)
        ej = float(wj @ hf[r])
        tj, to = _tol(hf[r], wj), _tol(hf[r], wo)
        assert ej >= top1[r] - (tj + to), (r, j, o, ej, top1[r], top2[r], tj, to)
        if top1[r] - top2[r] > tj + to:
            assert j == o, (r, j, o)
        assert abs(float(logit[r]) - ej) <= tj, (r, logit[r], ej, tj)
        exact += j == o
    assert exact >= min_exact * rows, (exact, rows)
    return o_idx


def test_lmhead_tiny_f16(cuda_dev):
    cfg = W.LMHEAD_TINY
    inp = W.generate_lmhead(cfg, seed=0)
    idx, lg, st, _ = _gpu(inp["hidden"], inp["weight"], cfg.dtype)
    assert st == 0
    _check(inp["hidden"], inp["weight"], cfg.dtype, idx, lg)


# every padded row count (16 .. 256) in both operand types, on a ragged
# vocabulary (5000 = 39 tiles of 128 + 8) and d_model = 320 (five 64-wide chunks)
@pytest.mark.parametrize("dtype", [W.BF16, W.F16])
@pytest.mark.parametrize("rows", [1, 16, 17, 40, 64, 65, 96, 100, 128, 150, 192, 256])
def test_lmhead_every_row_padding(cuda_dev, rows, dtype):
    cfg = W.LmHeadConfig(f"lmhead-pad-{rows}", rows=rows, d_model=320, vocab=5000, dtype=dtype)
    inp = W.generate_lmhead(cfg, seed=1)
    idx, lg, st, _ = _gpu(inp["hidden"], inp["weight"], dtype)
    assert st == 0
    _check(inp["hidden"], inp["weight"], dtype, idx, lg)


# fewer vocabulary tiles than SMs, a single partial tile, a single vocabulary row
@pytest.mark.parametrize("vocab", [1, 100, 128, 129, 1000])
def test_lmhead_small_vocabularies(cuda_dev, vocab):
    cfg = W.LmHeadConfig(f"lmhead-v{vocab}", rows=23, d_model=128, vocab=vocab, dtype=W.BF16)
    inp = W.generate_lmhead(cfg, seed=2)
    idx, lg, st, _ = _gpu(inp["hidden"], inp["weight"], W.BF16)
    assert st == 0
    _check(inp["hidden"], inp["weight"], W.BF16, idx, lg, min_exact=0.8)


def test_lmhead_planted_ties_go_to_the_lowest_index(cuda_dev):
    """Rows whose maximum sits on two identical weight rows (same lane of the
    128-row tile, in another CTA's range, or in the ragged last tile) must
    return the lower index; the two logits are bit-identical in any
    arithmetic, so this is exact."""
    cfg = W.LmHeadConfig("lmhead-ties", rows=23, d_model=512, vocab=30011, dtype=W.BF16)
    inp = W.generate_lmhead(cfg, seed=3)
    h, w = inp["hidden"], inp["weight"].copy()
    plants = {0: (5, 5 + 128), 1: (300, 300 + 128 * 150), 2: (7, 30010), 3: (29900, 30000), 22: (1000, 1001)}
    for r, (lo, hi) in plants.items():
        big = W.f32_to_bf16_bits(np.float32(0.05) * _f64(h[r], W.BF16).astype(np.float32))
        w[lo] = big
        w[hi] = big
    idx, lg, st, _ = _gpu(h, w, W.BF16)
    assert st == 0
    o_idx = _check(h, w, W.BF16, idx, lg)
    for r, (lo, _) in plants.items():
        assert o_idx[r] == lo and idx[r] == lo, (r, idx[r], o_idx[r])


def test_lmhead_workspace_reused_across_calls(cuda_dev):
    cfg = W.LmHeadConfig("lmhead-reuse", rows=41, d_model=256, vocab=7000, dtype=W.BF16)
    a = W.generate_lmhead(cfg, seed=4)
    b = W.generate_lmhead(cfg, seed=5)
    ia, la, sa, ws = _gpu(a["hidden"], a["weight"], W.BF16)
    ib, lb, sb, _ = _gpu(b["hidden"], b["weight"], W.BF16, reuse_ws=ws)
    ia2, la2, _, _ = _gpu(a["hidden"], a["weight"], W.BF16, reuse_ws=ws)
    assert sa == 0 and sb == 0
    assert np.array_equal(ia, ia2) and np.array_equal(la.view(np.uint32), la2.view(np.uint32))
    _check(b["hidden"], b["weight"], W.BF16, ib, lb)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [W.LMHEAD_27B_B22, W.LMHEAD_27B_B40], ids=lambda c: c.name)
def test_lmhead_full_vocabulary(cuda_dev, cfg):
    inp = W.generate_lmhead(cfg, seed=0)
    idx, lg, st, _ = _gpu(inp["hidden"], inp["weight"], cfg.dtype)
    assert st == 0
    _check(inp["hidden"], inp["weight"], cfg.dtype, idx, lg)
