"""lucetree_verify_attn_noalloc: the attention entry point for callers that
cannot allocate device memory (the library supplies a fixed 32 MiB scratch
array).  Two calls in a row, on different inputs, must each match the
workspace-taking entry point within the attention tolerance; oversized
shapes are refused before any launch.  This file is collected last."""
import numpy as np
import pytest

import workloads as W
from tests.helpers import ATTN_TOL, row_error, run_attention, to_device

pytestmark = pytest.mark.gpu


def _noalloc(d, cfg):
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    dev = d["q"].device
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    anc = torch.empty(cfg.B, cfg.N, dtype=torch.int64, device=dev)
    LT.lucetree_build_anc_mask(d["parent"], anc, status)
    out = torch.full((cfg.B, cfg.N, cfg.Hq, cfg.D), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((cfg.B, cfg.N, cfg.Hq), float("nan"), dtype=torch.float32, device=dev)
    LT.lucetree_verify_attn_noalloc(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"],
                                    d["v_tree"], anc, out, status, lse=lse)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


def test_noalloc_matches_workspace_entry_point_twice(cuda_dev):
    first = W.VerifyConfig("noalloc-a", ctx=(20000, 333), Hq=24, Hkv=4, D=256, dtype=W.BF16, N=22, tree="random",
                           branch_cap=4, vocab=64, paged="permuted", spare_pages=8)
    second = W.VerifyConfig("noalloc-b", ctx=(5000,), Hq=8, Hkv=2, D=128, dtype=W.F16, N=9, tree="random",
                            vocab=64, paged="permuted", spare_pages=2)
    for cfg in (first, second):
        inp = W.generate(cfg, seed=31)
        d = to_device(inp, cfg)
        ref, ref_lse, st_ref = run_attention(d, cfg, lse=True)
        got, got_lse, st = _noalloc(d, cfg)
        assert st == 0 and st_ref == 0
        g = got.cpu().numpy().reshape(-1, cfg.D)
        assert np.isfinite(g).all()
        assert row_error(g, ref.cpu().numpy().reshape(-1, cfg.D).astype(np.float64)).max() <= ATTN_TOL
        assert np.allclose(got_lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=1e-5, atol=1e-5)


def test_noalloc_refuses_sizes_past_its_scratch(cuda_dev):
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    B, N, Hq, Hkv, D = 64, 64, 32, 8, 256
    assert LT.lucetree_verify_attn_workspace(B, N, Hq, Hkv, D) > LT.NOALLOC_SCRATCH_BYTES
    # the C entry point itself refuses, before touching any pointer
    lib = LT.load()
    a = LT.AttnArgs()
    a.dtype, a.B, a.N, a.Hq, a.Hkv, a.D, a.page_size, a.scale = 1, B, N, Hq, Hkv, D, 64, 0.0625
    assert lib.lucetree_verify_attn_noalloc(a, None) == 3  # LUCETREE_ERR_WORKSPACE
    # and so does the binding
    q = torch.zeros(B, N, Hq, D, dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros(1, Hkv, 64, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(LT.LucetreeError):
        LT.lucetree_verify_attn_noalloc(q, kp, kp, None, None, None, None, None, None, None)
