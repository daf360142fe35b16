"""Tree-aware recurrent-state (gated delta rule) step and its commit through
the C-ABI against the fp64 oracle.

The kernel keeps the state in fp32.  Each node adds one update of the state
(a dk-term dot product, a scale and a rank-1 term) on top of its parent's, and
every factor is contractive (alpha <= 1, |I - beta k k^T| <= 1 for unit k and
beta in [0, 1]).  To first order the rounding error of node i's output
therefore stays within (depth_i + 1) * (dk + 4) * 2^-24 of the largest output
of its row; the tests allow four times that.  A commit of nothing must leave
the state bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


def _lt():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    return LT


def _odt(cfg):
    return oracle.BF16 if cfg.dtype == W.BF16 else oracle.F16


def _dev(inp, cfg):
    import torch
    tdt = torch.bfloat16 if cfg.dtype == W.BF16 else torch.float16
    d = {}
    for key in ("q", "k", "v"):
        d[key] = torch.from_numpy(np.ascontiguousarray(inp[key]).view(np.int16)).view(tdt).cuda()
    for key in ("alpha", "beta", "state"):
        d[key] = torch.from_numpy(np.ascontiguousarray(inp[key])).cuda()
    d["parent"] = torch.from_numpy(np.ascontiguousarray(inp["parent"])).cuda()
    return d


def _depths(parent):
    dep = np.zeros(parent.shape, np.int64)
    for b in range(parent.shape[0]):
        for i in range(parent.shape[1]):
            p = parent[b, i]
            dep[b, i] = 0 if p < 0 else dep[b, p] + 1
    return dep


def _tree(cfg, inp):
    import torch
    LT = _lt()
    d = _dev(inp, cfg)
    out = torch.full((cfg.B, cfg.N, cfg.Hv, cfg.dv), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["state"], out, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), st.item(), d


def _check_tree(cfg, inp):
    got, status, d = _tree(cfg, inp)
    assert status == 0
    ref = oracle.delta_tree(inp, _odt(cfg))
    dep = _depths(inp["parent"])
    tol = 4.0 * (dep + 1) * (cfg.dk + 4) * 2.0 ** -24            # [B][N]
    err = np.abs(got - ref).max(axis=-1) / np.abs(ref).max(axis=-1)  # [B][N][Hv]
    assert np.isfinite(got).all()
    worst = (err / tol[:, :, None]).max()
    assert worst <= 1.0, f"worst error {worst:.2f} x tolerance"
    # the state is only read
    assert np.array_equal(d["state"].cpu().numpy(), inp["state"])
    return err


@pytest.mark.parametrize("cfg", [W.DELTA_TINY, W.DELTA_27B_B22, W.DELTA_27B_B40, W.DELTA_27B_B64_CHAIN],
                         ids=lambda c: c.name)
def test_delta_tree_matches_oracle(cuda_dev, cfg):
    _check_tree(cfg, W.generate_delta(cfg, seed=0))


@pytest.mark.parametrize("N,tree", [(1, "chain"), (5, "random"), (26, "random"), (27, "random"), (64, "random")])
def test_delta_tree_batches_and_column_splits(cuda_dev, N, tree):
    # B = 3 different trees; N = 26 / 27 straddle the 8 -> 4 column split
    cfg = W.DeltaConfig(f"delta-b3-{N}-{tree}", B=3, N=N, Hk=2, Hv=6, dv=64, dtype=W.BF16, tree=tree, branch_cap=3)
    _check_tree(cfg, W.generate_delta(cfg, seed=N))


def test_delta_tree_flags_bad_parent(cuda_dev):
    LT = _lt()
    cfg = W.DeltaConfig("delta-bad", B=1, N=6, Hk=1, Hv=2, dv=16, dtype=W.F16)
    inp = W.generate_delta(cfg, seed=2)
    inp["parent"] = np.array([[-1, 0, 5, 1, 1, 2]], np.int32)
    _, status, _ = _tree(cfg, inp)
    assert status & LT.DEV_BAD_PARENT


def _commit(cfg, inp, acc, lens):
    import torch
    LT = _lt()
    d = _dev(inp, cfg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    LT.lucetree_delta_commit(d["k"], d["v"], d["alpha"], d["beta"], torch.from_numpy(acc).cuda(),
                             torch.from_numpy(lens).cuda(), d["state"], st)
    torch.cuda.synchronize()
    return d["state"].cpu().numpy(), st.item()


def _root_path(parent, i):
    path = []
    while i >= 0:
        path.append(i)
        i = parent[i]
    return path[::-1]


@pytest.mark.parametrize("cfg", [W.DELTA_TINY, W.DELTA_27B_B22, W.DELTA_27B_B64_CHAIN], ids=lambda c: c.name)
def test_delta_commit_matches_oracle(cuda_dev, cfg):
    inp = W.generate_delta(cfg, seed=1)
    rng = np.random.default_rng(9)
    acc = np.full((cfg.B, cfg.N), -1, np.int32)
    lens = np.zeros(cfg.B, np.int32)
    for b in range(cfg.B):
        path = _root_path(inp["parent"][b], int(rng.integers(0, cfg.N)))
        acc[b, :len(path)] = path
        lens[b] = len(path)
    got, status = _commit(cfg, inp, acc, lens)
    assert status == 0
    ref = oracle.delta_commit(inp, _odt(cfg), acc, lens)
    tol = 4.0 * (lens.max() + 1) * (cfg.dk + 4) * 2.0 ** -24
    assert np.abs(got - ref).max() <= tol * np.abs(ref).max()


def test_delta_commit_of_nothing_keeps_the_state_and_bad_nodes_are_flagged(cuda_dev):
    LT = _lt()
    cfg = W.DeltaConfig("delta-c0", B=2, N=8, Hk=1, Hv=2, dv=32, dtype=W.BF16)
    inp = W.generate_delta(cfg, seed=3)
    got, status = _commit(cfg, inp, np.zeros((2, 8), np.int32), np.zeros(2, np.int32))
    assert status == 0 and np.array_equal(got, inp["state"])
    acc = np.zeros((2, 8), np.int32)
    acc[0, :2] = [0, 9]
    got, status = _commit(cfg, inp, acc, np.array([2, 0], np.int32))
    assert status & LT.DEV_BAD_NODE
    assert np.array_equal(got, inp["state"])


def test_delta_tree_then_commit_reads_back_the_accepted_output(cuda_dev):
    # after committing node i's path, S^T q_i is node i's tree-pass output
    import torch
    cfg = W.DeltaConfig("delta-rb", B=1, N=22, Hk=2, Hv=4, dv=128, dtype=W.BF16, tree="random", branch_cap=4)
    inp = W.generate_delta(cfg, seed=4)
    out, status, _ = _tree(cfg, inp)
    i = 21
    path = _root_path(inp["parent"][0], i)
    acc = np.full((1, cfg.N), -1, np.int32)
    acc[0, :len(path)] = path
    st, status2 = _commit(cfg, inp, acc, np.array([len(path)], np.int32))
    assert status == 0 and status2 == 0
    q = inp["q"].view(np.uint16)
    qf = ((q.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)
    for h in range(cfg.Hv):
        back = qf[0, i, h // 2] @ st[0, h].astype(np.float64)
        assert np.abs(back - out[0, i, h]).max() <= 1e-4 * np.abs(out[0, i, h]).max()
