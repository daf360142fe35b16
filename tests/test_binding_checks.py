"""The Python binding's shape and element-type checks, on the CPU.

The library is replaced by a stub whose entry points return LUCETREE_OK, so
every wrapper runs its marshalling without a GPU.  Two directions:
the tensors that the tests, the bench and the smoke run build for each call
(same generators, same dtypes) pass; a tensor whose shape or element type
would make a kernel index past its end is refused with LucetreeError before
any call is made."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
from tests.helpers import to_device


class _StubLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def entry(*args):
            self.calls.append(name)
            return LT.LUCETREE_OK
        return entry


@pytest.fixture
def stub(monkeypatch):
    lib = _StubLib()
    monkeypatch.setattr(LT, "load", lambda path=None: lib)
    monkeypatch.setattr(LT, "_ptr", lambda t: None if t is None else ctypes.c_void_p(t.data_ptr()))
    monkeypatch.setattr(LT, "_host_ptr", lambda t: ctypes.c_void_p(t.data_ptr()))
    monkeypatch.setattr(LT, "_stream", lambda s: ctypes.c_void_p(0))
    return lib


CFG = W.VerifyConfig("binding", ctx=(100, 0, 700), Hq=6, Hkv=2, D=256, dtype=W.BF16, N=5, tree="random",
                     branch_cap=3, vocab=300, paged="permuted", spare_pages=2)


@pytest.fixture(scope="module")
def attn():
    inp = W.generate(CFG, seed=3)
    d = to_device(inp, CFG, device="cpu")
    B, N, Hq, D = CFG.B, CFG.N, CFG.Hq, CFG.D
    extra = dict(anc=torch.empty(B, N, dtype=torch.int64), out=torch.empty(B, N, Hq, D, dtype=torch.float32),
                 lse=torch.empty(B, N, Hq, dtype=torch.float32), status=torch.zeros(1, dtype=torch.int32),
                 ws=torch.empty(256, dtype=torch.uint8))
    return inp, d, extra


def _verify(d, x, **over):
    a = dict(q=d["q"], k_pool=d["k_pool"], v_pool=d["v_pool"], page_table=d["page_table"], ctx_len=d["ctx_len"],
             k_tree=d["k_tree"], v_tree=d["v_tree"], anc_mask=x["anc"], out=x["out"], status=x["status"],
             workspace=x["ws"], lse=x["lse"])
    a.update(over)
    LT.lucetree_verify_attn(**a)


def test_verify_attn_accepts_generated_inputs(stub, attn):
    _, d, x = attn
    _verify(d, x)
    _verify(d, x, lse=None)
    assert stub.calls == ["lucetree_verify_attn"] * 2


@pytest.mark.parametrize("field,bad", [
    ("out", lambda d, x: x["out"].to(torch.bfloat16)),                      # fp32 written into a 2-byte buffer
    ("out", lambda d, x: x["out"][:, :-1].contiguous()),                    # one node short
    ("lse", lambda d, x: x["lse"][..., :-1].contiguous()),
    ("anc_mask", lambda d, x: x["anc"].to(torch.int32)),                    # 64-bit masks read from 4-byte words
    ("page_table", lambda d, x: d["page_table"].to(torch.int64)),
    ("page_table", lambda d, x: d["page_table"].reshape(-1)),
    ("ctx_len", lambda d, x: d["ctx_len"][:-1].contiguous()),
    ("v_pool", lambda d, x: d["v_pool"][:-1].contiguous()),                 # fewer pages than k_pool
    ("v_pool", lambda d, x: d["v_pool"].to(torch.float16)),                 # dtype differs from q
    ("k_tree", lambda d, x: d["k_tree"][:, :, :1].contiguous()),            # one KV head
    ("q", lambda d, x: d["q"][..., :128].contiguous()),                     # head dim differs from the pools
    ("status", lambda d, x: torch.zeros(0, dtype=torch.int32)),
    ("anc_mask", lambda d, x: None),
])
def test_verify_attn_refuses_mismatches(stub, attn, field, bad):
    _, d, x = attn
    with pytest.raises(LT.LucetreeError):
        _verify(d, x, **{field: bad(d, x)})
    assert stub.calls == []


@pytest.mark.parametrize("v_format", [W.V_INT8, W.V_INT4], ids=["int8", "int4"])
def test_verify_attn_vq_shapes(stub, attn, v_format):
    _, d, x = attn
    vq = W.generate_vq(CFG, v_format, seed=3)
    codes, vexp = torch.from_numpy(vq["v_codes"]), torch.from_numpy(vq["v_exp"])

    def call(c, e, fmt=v_format):
        LT.lucetree_verify_attn_vq(d["q"], d["k_pool"], c, e, fmt, d["page_table"], d["ctx_len"], d["k_tree"],
                                   d["v_tree"], x["anc"], x["out"], x["status"], x["ws"])

    call(codes, vexp)
    assert stub.calls == ["lucetree_verify_attn_vq"]
    other = W.V_INT4 if v_format == W.V_INT8 else W.V_INT8
    for c, e, fmt in ((codes, vexp, other),                              # code row width of the other format
                      (codes, vexp[:, :, :-1].contiguous(), v_format),   # exponents short of a page
                      (codes.view(torch.int8)[:-1].contiguous(), vexp, v_format),
                      (codes, vexp, 7)):
        with pytest.raises(LT.LucetreeError):
            call(c, e, fmt)
    assert stub.calls == ["lucetree_verify_attn_vq"]


def test_noalloc_uses_the_same_checks(stub, attn):
    _, d, x = attn
    LT.lucetree_verify_attn_noalloc(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"],
                                    d["v_tree"], x["anc"], x["out"], x["status"], lse=x["lse"])
    with pytest.raises(LT.LucetreeError):
        LT.lucetree_verify_attn_noalloc(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"],
                                        d["k_tree"], d["v_tree"], x["anc"], x["out"].half(), x["status"])
    assert stub.calls.count("lucetree_verify_attn_noalloc") == 1


def test_tree_ops_accept_generated_inputs_and_refuse_mismatches(stub, attn):
    inp, d, x = attn
    B, N = CFG.B, CFG.N
    st = x["status"]
    LT.lucetree_build_anc_mask(d["parent"], x["anc"], st)
    am = torch.empty(B, N + 1, dtype=torch.int32)
    LT.lucetree_argmax(d["logits"], am, x["ws"])
    acc, alen, bonus = (torch.empty(B, N, dtype=torch.int32), torch.empty(B, dtype=torch.int32),
                        torch.empty(B, dtype=torch.int32))
    LT.lucetree_accept(d["parent"], d["draft"], am, CFG.vocab, acc, alen, bonus, st)
    o_acc, o_len, _ = oracle.accept(inp["parent"], inp["draft"], oracle.argmax(inp["logits"]))
    ctx_out = torch.empty_like(d["ctx_len"])
    LT.lucetree_commit(d["k_tree"], d["v_tree"], torch.from_numpy(o_acc), torch.from_numpy(o_len), d["page_table"],
                       d["ctx_len"], ctx_out, d["k_pool"], d["v_pool"], st)
    LT.lucetree_commit(d["k_tree"], d["v_tree"], acc, alen, d["page_table"], d["ctx_len"], d["ctx_len"],
                       d["k_pool"], d["v_pool"], st)  # ctx_len updated in place
    good = ["lucetree_build_anc_mask", "lucetree_argmax", "lucetree_accept", "lucetree_commit", "lucetree_commit"]
    assert stub.calls == good

    refused = [
        lambda: LT.lucetree_build_anc_mask(d["parent"].to(torch.int64), x["anc"], st),
        lambda: LT.lucetree_build_anc_mask(d["parent"], x["anc"][:, :-1].contiguous(), st),
        lambda: LT.lucetree_argmax(d["logits"], am[:, :-1].contiguous(), x["ws"]),
        lambda: LT.lucetree_argmax(d["logits"].double(), am, x["ws"]),
        lambda: LT.lucetree_accept(d["parent"], d["draft"], am[:, :-1].contiguous(), CFG.vocab, acc, alen, bonus, st),
        lambda: LT.lucetree_accept(d["parent"], d["draft"].to(torch.int64), am, CFG.vocab, acc, alen, bonus, st),
        lambda: LT.lucetree_commit(d["k_tree"], d["v_tree"], acc, alen, d["page_table"], d["ctx_len"], ctx_out,
                                   d["k_pool"], d["v_pool"][:-1].contiguous(), st),
        lambda: LT.lucetree_commit(d["k_tree"], d["v_tree"][:, :-1].contiguous(), acc, alen, d["page_table"],
                                   d["ctx_len"], ctx_out, d["k_pool"], d["v_pool"], st),
        lambda: LT.lucetree_commit(d["k_tree"], d["v_tree"], acc.to(torch.int64), alen, d["page_table"],
                                   d["ctx_len"], ctx_out, d["k_pool"], d["v_pool"], st),
    ]
    for call in refused:
        with pytest.raises(LT.LucetreeError):
            call()
    assert stub.calls == good


def test_verify_step_buffers_pass_the_checks(stub, attn):
    _, d, _ = attn
    step = LT.VerifyStep(CFG.B, CFG.N, CFG.Hq, CFG.Hkv, CFG.D, CFG.vocab, device="cpu")
    args = (d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"], d["v_tree"], d["parent"],
            d["draft"], d["logits"])
    step.run(*args)
    step.run(*args)
    assert stub.calls[-2:] == ["lucetree_verify_step"] * 2
    assert len(step._packed) == 1  # the second call reused the checked arguments
    step.run_calls(*args)
    assert stub.calls[-5:] == ["lucetree_build_anc_mask", "lucetree_verify_attn", "lucetree_argmax",
                               "lucetree_accept", "lucetree_commit"]


def test_verify_step_refuses_mismatched_buffers(stub, attn):
    _, d, _ = attn
    step = LT.VerifyStep(CFG.B, CFG.N, CFG.Hq, CFG.Hkv, CFG.D, CFG.vocab, device="cpu")
    good = dict(q=d["q"], k_pool=d["k_pool"], v_pool=d["v_pool"], page_table=d["page_table"], ctx_len=d["ctx_len"],
                k_tree=d["k_tree"], v_tree=d["v_tree"], parent=d["parent"], draft=d["draft"], logits=d["logits"])
    for k, bad in (("logits", d["logits"][:, :-1].contiguous()),      # one row short per sequence
                   ("draft", d["draft"].to(torch.int64)),              # wrong element type
                   ("parent", d["parent"][:-1].contiguous()),          # one sequence short
                   ("k_tree", d["k_tree"].view(torch.float16))):       # dtype differs from q
        with pytest.raises(LT.LucetreeError):
            step.run(**dict(good, **{k: bad}))
    assert "lucetree_verify_step" not in stub.calls


def test_lmhead_shapes(stub):
    lc = W.LMHEAD_TINY
    inp = W.generate_lmhead(lc, seed=0)
    h = torch.from_numpy(np.ascontiguousarray(inp["hidden"]).view(np.int16)).view(torch.float16)
    w = torch.from_numpy(np.ascontiguousarray(inp["weight"]).view(np.int16)).view(torch.float16)
    out, lg, st = (torch.empty(lc.rows, dtype=torch.int32), torch.empty(lc.rows, dtype=torch.float32),
                   torch.zeros(1, dtype=torch.int32))
    ws = torch.empty(256, dtype=torch.uint8)
    LT.lucetree_lmhead_argmax(h, w, out, st, ws, out_logit=lg)
    LT.lucetree_lmhead_argmax(h, w, out, st, ws)
    assert stub.calls == ["lucetree_lmhead_argmax"] * 2
    for args in ((h, w[:, :-64].contiguous(), out, st, ws),     # d_model differs
                 (h, w.view(torch.bfloat16), out, st, ws),        # dtype differs
                 (h, w, out[:-1].contiguous(), st, ws)):          # one index short
        with pytest.raises(LT.LucetreeError):
            LT.lucetree_lmhead_argmax(*args)
    with pytest.raises(LT.LucetreeError):
        LT.lucetree_lmhead_argmax(h, w, out, st, ws, out_logit=lg.half())
    assert stub.calls == ["lucetree_lmhead_argmax"] * 2


def test_delta_shapes(stub):
    dc = W.DELTA_TINY
    inp = W.generate_delta(dc, seed=0)
    d = {k: torch.from_numpy(np.ascontiguousarray(inp[k]).view(np.int16)).view(torch.float16) for k in "qkv"}
    for k in ("alpha", "beta", "state", "parent"):
        d[k] = torch.from_numpy(np.ascontiguousarray(inp[k]))
    out = torch.empty(dc.B, dc.N, dc.Hv, dc.dv, dtype=torch.float32)
    st = torch.zeros(1, dtype=torch.int32)
    acc = torch.full((dc.B, dc.N), -1, dtype=torch.int32)
    alen = torch.zeros(dc.B, dtype=torch.int32)
    LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["state"], out, st)
    LT.lucetree_delta_commit(d["k"], d["v"], d["alpha"], d["beta"], acc, alen, d["state"], st)
    assert stub.calls == ["lucetree_delta_tree", "lucetree_delta_commit"]
    refused = [
        lambda: LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"],
                                       d["state"][..., :-8].contiguous(), out, st),
        lambda: LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"].double(), d["beta"], d["parent"],
                                       d["state"], out, st),
        lambda: LT.lucetree_delta_tree(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["parent"], d["state"],
                                       out[:, :-1].contiguous(), st),
        lambda: LT.lucetree_delta_tree(d["q"].view(torch.bfloat16), d["k"], d["v"], d["alpha"], d["beta"],
                                       d["parent"], d["state"], out, st),
        lambda: LT.lucetree_delta_commit(d["k"], d["v"], d["alpha"], d["beta"], acc[:, :-1].contiguous(), alen,
                                         d["state"], st),
        lambda: LT.lucetree_delta_commit(d["k"], d["v"], d["alpha"], d["beta"], acc, None, d["state"], st),
    ]
    for call in refused:
        with pytest.raises(LT.LucetreeError):
            call()
    assert stub.calls == ["lucetree_delta_tree", "lucetree_delta_commit"]


def test_stage_shapes(stub):
    hk = torch.zeros(2, 2, 64, 8, dtype=torch.int16)
    pk = torch.zeros(3, 2, 64, 8, dtype=torch.int16)
    idx = torch.tensor([1, 0], dtype=torch.int32)
    st = torch.zeros(1, dtype=torch.int32)
    table = torch.full((2, 4), -1, dtype=torch.int32)
    LT.lucetree_stage_pages(hk, hk.clone(), idx, idx, pk, pk.clone(), st)
    LT.lucetree_stage_pages(hk, hk.clone(), idx, idx, pk, pk.clone(), st, table_idx=idx, page_table=table)
    LT.lucetree_stage_pages(hk.view(torch.bfloat16), hk.view(torch.bfloat16), idx[:0], idx[:0], pk, pk, st)
    assert stub.calls == ["lucetree_stage_pages"] * 3
    refused = [
        lambda: LT.lucetree_stage_pages(hk, hk[:1].contiguous(), idx, idx, pk, pk, st),       # host_v shorter
        lambda: LT.lucetree_stage_pages(hk, hk, idx, idx, pk, pk[..., :4].contiguous(), st),  # pool geometry
        lambda: LT.lucetree_stage_pages(hk.float(), hk.float(), idx, idx, pk, pk, st),         # 4-byte host data
        lambda: LT.lucetree_stage_pages(hk, hk, idx, idx[:1].contiguous(), pk, pk, st),        # dst count
        lambda: LT.lucetree_stage_pages(hk, hk, idx, idx, pk, pk, st, table_idx=idx),          # no table
        lambda: LT.lucetree_stage_pages(hk, hk, idx.long(), idx, pk, pk, st),
    ]
    for call in refused:
        with pytest.raises(LT.LucetreeError):
            call()
    assert stub.calls == ["lucetree_stage_pages"] * 3
