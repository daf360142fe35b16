"""The failure path of the bounded waits, made to run on purpose: a wait on a
barrier that nothing arrives on gives up after its cycle limit, the status
word carries LUCETREE_DEV_TIMEOUT, and the context stays usable (a verify
step right after still matches the oracle)."""
import numpy as np
import pytest

import oracle
import workloads as W
from tests.helpers import ATTN_TOL, oracle_dtype, row_error, run_attention, to_device

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_the_context_survives(cuda_dev):
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 20_000_000  # about 10 ms of SM cycles
    LT.lucetree_selftest_wait_timeout(status, limit, waited)
    torch.cuda.synchronize()
    assert status.item() == LT.DEV_TIMEOUT
    assert limit < waited.item() < 50 * limit

    cfg = W.TINY
    inp = W.generate(cfg, seed=0)
    out, _, st = run_attention(to_device(inp, cfg), cfg)
    assert st == 0
    ref, _ = oracle.verify_attn(inp, oracle_dtype(cfg))
    assert row_error(out.cpu().numpy().reshape(ref.shape), ref).max() <= ATTN_TOL
