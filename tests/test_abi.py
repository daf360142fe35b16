"""The C-ABI library loads without a GPU and exports every symbol the header
declares; the binding refuses host tensors.  No compute calls here."""
import ctypes
import os
import re

import pytest

from speculative_decoding_tree_ddtree_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names.update(re.findall(r"^LUCETREE_API\s+[\w\s\*]+?\b(lucetree_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_calls():
    d = _declared()
    for name in ("lucetree_verify_attn", "lucetree_argmax", "lucetree_accept", "lucetree_commit"):
        assert name in d


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_lists_every_declared_symbol():
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    assert set(_declared()) <= set(LT.EXPORTED)


def test_host_side_queries_without_gpu(lib):
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    lt = LT.load()
    assert lt.lucetree_abi_version() == 1
    assert lt.lucetree_status_string(3) == b"workspace missing or too small"
    n = ctypes.c_size_t(0)
    # unsupported head dim and budget are rejected before any device work
    assert lt.lucetree_verify_attn_workspace(1, 22, 24, 4, 96, ctypes.byref(n)) == 2
    assert lt.lucetree_verify_attn_workspace(1, 65, 24, 4, 256, ctypes.byref(n)) == 2
    assert lt.lucetree_verify_attn_workspace(1, 22, 24, 5, 256, ctypes.byref(n)) == 2
    assert lt.lucetree_accept(None, None, None, 1, 1, 1, None, None, None, None, None) == 1
    assert lt.lucetree_verify_attn(None, None, 0, None) == 1
    assert lt.lucetree_commit(None, None) == 1
    # lm_head + argmax: row count and d_model limits, checked on the host
    assert lt.lucetree_lmhead_argmax_workspace(0, ctypes.byref(n)) == 1
    assert lt.lucetree_lmhead_argmax_workspace(257, ctypes.byref(n)) == 2
    assert lt.lucetree_lmhead_argmax_workspace(23, ctypes.byref(n)) == 0 and n.value >= 23 * 8 + 4
    assert lt.lucetree_lmhead_argmax(None, None, 0, None) == 1
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    for rows, d_model, want in ((300, 256, 2), (8, 100, 2), (0, 256, 1)):
        a = LT.LmHeadArgs(dtype=LT.LUCETREE_BF16, rows=rows, d_model=d_model, vocab=1000,
                          hidden=fake, weight=fake, out_idx=fake, out_logit=None, status=fake)
        assert lt.lucetree_lmhead_argmax(ctypes.byref(a), None, 0, None) == want
    a = LT.LmHeadArgs(dtype=LT.LUCETREE_BF16, rows=8, d_model=256, vocab=1000,
                      hidden=fake, weight=fake, out_idx=fake, out_logit=None, status=fake)
    assert lt.lucetree_lmhead_argmax(ctypes.byref(a), None, 0, None) == 3  # no workspace
    # quantised-V attention: format and head dim are checked on the host
    aa = LT.AttnArgs()
    aa.dtype, aa.B, aa.N, aa.Hq, aa.Hkv, aa.D, aa.page_size = LT.LUCETREE_BF16, 1, 4, 4, 1, 256, 64
    assert lt.lucetree_verify_attn_vq(ctypes.byref(aa), 3, fake, None, 0, None) == 2   # unknown format
    assert lt.lucetree_verify_attn_vq(ctypes.byref(aa), 1, None, None, 0, None) == 1   # no exponents
    aa.D = 128
    assert lt.lucetree_verify_attn_vq(ctypes.byref(aa), 1, fake, None, 0, None) == 2   # head dim 256 only
    # delta-rule step: shape limits and required pointers, checked on the host
    assert lt.lucetree_delta_tree(None, None) == 1 and lt.lucetree_delta_commit(None, None) == 1
    for (dk, dv, N, want) in ((64, 128, 8, 2), (128, 12, 8, 2), (128, 128, 65, 2), (128, 128, 0, 1)):
        d = LT.DeltaArgs(dtype=LT.LUCETREE_BF16, B=1, N=N, Hk=1, Hv=2, dk=dk, dv=dv, q=fake, k=fake, v=fake,
                         alpha=fake, beta=fake, parent=fake, state=fake, out=fake, status=fake)
        assert lt.lucetree_delta_tree(ctypes.byref(d), None) == want
    d = LT.DeltaArgs(dtype=LT.LUCETREE_BF16, B=1, N=8, Hk=1, Hv=2, dk=128, dv=128, k=fake, v=fake,
                     alpha=fake, beta=fake, state=fake, status=fake)
    assert lt.lucetree_delta_commit(ctypes.byref(d), None) == 1  # no accepted path given
    # host-resident page staging: sizes and pointers are checked before any CUDA call
    assert lt.lucetree_stage_pages(None, None) == 1
    ok = dict(Hkv=2, D=128, n=3, host_k=fake, host_v=fake, host_pages=4, src=fake, dst=fake, table_idx=None,
              page_table=None, table_len=0, k_pool=fake, v_pool=fake, num_pages=8, status=fake)
    for change in (dict(n=-1), dict(D=100), dict(Hkv=0), dict(num_pages=0), dict(host_v=None),
                   dict(host_k=fake + 8), dict(table_idx=fake), dict(status=None)):
        st = LT.StageArgs(**{**ok, **change})
        assert lt.lucetree_stage_pages(ctypes.byref(st), None) == 1, change
    st = LT.StageArgs(**{**ok, "n": 0, "host_k": None})
    assert lt.lucetree_stage_pages(ctypes.byref(st), None) == 0  # nothing to stage: no launch, no error
    # the wait-timeout self-test: status required, limit within (0, 4e9]
    assert lt.lucetree_selftest_wait_timeout(None, 1000, None, None) == 1
    assert lt.lucetree_selftest_wait_timeout(fake, 0, None, None) == 1
    assert lt.lucetree_selftest_wait_timeout(fake, 4000000001, None, None) == 1


def test_binding_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    with pytest.raises(LT.LucetreeError):
        LT._ptr(torch.zeros(4))


def test_noalloc_scratch_size_matches_header():
    """The binding refuses oversized shapes before calling the library; its
    limit must be the header's LUCETREE_NOALLOC_SCRATCH_BYTES."""
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    src = open(os.path.join(ROOT, "include", "lucetree.h")).read()
    m = re.search(r"#define\s+LUCETREE_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "LUCETREE_NOALLOC_SCRATCH_BYTES not found"
    assert LT.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
