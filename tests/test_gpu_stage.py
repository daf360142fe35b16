"""Host-resident cold pages staged into the device pool through the C-ABI:
byte-exact against the oracle's copy, and attention over the staged pages
matches the oracle on the logical cache."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import ATTN_TOL, oracle_dtype, row_error, run_attention, to_device

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_stage_pages_is_byte_exact(cuda_dev):
    import torch
    LT = _lt()
    rng = np.random.default_rng(0)
    Hkv, D, host_pages, num_pages = 3, 128, 40, 50
    host_k = rng.integers(0, 1 << 16, size=(host_pages, Hkv, 64, D), dtype=np.uint16)
    host_v = rng.integers(0, 1 << 16, size=(host_pages, Hkv, 64, D), dtype=np.uint16)
    pool_k = rng.integers(0, 1 << 16, size=(num_pages, Hkv, 64, D), dtype=np.uint16)
    pool_v = rng.integers(0, 1 << 16, size=(num_pages, Hkv, 64, D), dtype=np.uint16)
    src = rng.choice(host_pages, size=17, replace=False).astype(np.int32)
    dst = rng.choice(num_pages, size=17, replace=False).astype(np.int32)
    table = rng.integers(-1, num_pages, size=(4, 20)).astype(np.int32)
    tidx = rng.choice(table.size, size=17, replace=False).astype(np.int32)
    dk, dv = _t(pool_k.view(np.int16)), _t(pool_v.view(np.int16))
    dt = _t(table)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_stage_pages(_pinned(host_k), _pinned(host_v), _t(src), _t(dst), dk, dv, st, table_idx=_t(tidx),
                            page_table=dt)
    torch.cuda.synchronize()
    kp, vp, pt = oracle.stage_pages(host_k, host_v, src, dst, pool_k, pool_v, table_idx=tidx, page_table=table)
    assert st.item() == 0
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), vp)
    assert np.array_equal(dt.cpu().numpy(), pt)


def test_stage_pages_flags_and_skips_bad_ids(cuda_dev):
    import torch
    LT = _lt()
    host = np.ones((2, 1, 64, 8), np.uint16)
    pool = np.zeros((3, 1, 64, 8), np.uint16)
    dk, dv = _t(pool.view(np.int16)), _t(pool.view(np.int16))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_stage_pages(_pinned(host), _pinned(host), _t(np.array([0, 5], np.int32)),
                            _t(np.array([1, 2], np.int32)), dk, dv, st)
    torch.cuda.synchronize()
    assert st.item() & LT.DEV_BAD_PAGE
    got = dk.cpu().numpy().view(np.uint16)
    assert (got[1] == 1).all() and (got[2] == 0).all() and (got[0] == 0).all()


def test_stage_pages_refuses_pageable_host_memory(cuda_dev):
    import torch
    LT = _lt()
    host = torch.zeros(2, 1, 64, 8, dtype=torch.int16)  # not page-locked
    pool = torch.zeros(3, 1, 64, 8, dtype=torch.int16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(LT.LucetreeError):
        LT.lucetree_stage_pages(host, host, idx, idx, pool, pool, st)


def test_attention_over_staged_cold_pages(cuda_dev):
    # a third of the committed pages live in host pools; their device copies
    # are poisoned, they are staged into spare pages and the table repointed
    import torch
    LT = _lt()
    cfg = W.VerifyConfig("cold", ctx=(1500, 700, 2100), Hq=12, Hkv=3, D=128, dtype=W.BF16, N=7, tree="random",
                         branch_cap=3, vocab=256, paged="permuted", spare_pages=40)
    inp = W.generate(cfg, seed=11)
    pt = inp["page_table"]
    used = set(int(x) for x in pt[pt >= 0])
    spare = np.array(sorted(set(range(inp["k_pool"].shape[0])) - used), np.int32)
    rng = np.random.default_rng(5)
    cold_pos = np.array([i for i in range(pt.size) if pt.flat[i] >= 0 and rng.random() < 0.33], np.int32)
    cold_pages = pt.reshape(-1)[cold_pos]
    host_k = inp["k_pool"][cold_pages].copy()
    host_v = inp["v_pool"][cold_pages].copy()
    dst = spare[:len(cold_pos)]
    assert len(dst) == len(cold_pos) > 4
    d = to_device(inp, cfg)
    nan = W.NAN_BITS[cfg.dtype]
    poison = torch.tensor(int(np.uint16(nan).view(np.int16)), dtype=torch.int16)
    for which in ("k_pool", "v_pool"):  # the device copies of cold pages hold garbage
        d[which][torch.from_numpy(cold_pages.astype(np.int64)).cuda()] = poison.view(d[which].dtype).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_stage_pages(_pinned(host_k), _pinned(host_v), _t(np.arange(len(dst), dtype=np.int32)), _t(dst),
                            d["k_pool"], d["v_pool"], st, table_idx=_t(cold_pos), page_table=d["page_table"])
    out, _, status = run_attention(d, cfg)
    assert st.item() == 0 and status == 0
    ref, _ = oracle.verify_attn(inp, oracle_dtype(cfg))
    err = row_error(out.cpu().numpy().reshape(ref.shape), ref)
    assert err.max() <= ATTN_TOL
