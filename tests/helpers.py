"""Shared test plumbing: generated inputs to device tensors, the library calls
of one verify step, and the attention error metric."""
import functools

import numpy as np

import workloads as W

ATTN_TOL = 2e-3  # max over rows of max_d |gpu - oracle| / max_d |oracle|


def row_error(gpu: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per output row: max_d |gpu - ref| / max_d |ref|."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape)
    num = np.abs(gpu - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    return num / den


@functools.lru_cache(maxsize=4)
def cached_inputs(cfg: W.VerifyConfig, seed: int = 0, fill_unused: str = "nan"):
    return W.generate(cfg, seed=seed, fill_unused=fill_unused)


def oracle_dtype(cfg):
    import oracle
    return oracle.BF16 if cfg.dtype == W.BF16 else oracle.F16


def to_device(inp: dict, cfg: W.VerifyConfig, device="cuda"):
    import torch
    tdt = torch.bfloat16 if cfg.dtype == W.BF16 else torch.float16

    def h16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt).to(device)

    d = dict(
        q=h16(inp["q"]), k_pool=h16(inp["k_pool"]), v_pool=h16(inp["v_pool"]),
        k_tree=h16(inp["k_tree"]), v_tree=h16(inp["v_tree"]),
        page_table=torch.from_numpy(inp["page_table"]).to(device),
        ctx_len=torch.from_numpy(inp["ctx_len"]).to(device),
        parent=torch.from_numpy(inp["parent"]).to(device),
        draft=torch.from_numpy(inp["draft"]).to(device),
    )
    if inp.get("logits") is not None:
        d["logits"] = torch.from_numpy(inp["logits"]).to(device)
    return d


def bits16(t):
    """Device 16-bit tensor -> numpy uint16 bits."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_attention(d: dict, cfg: W.VerifyConfig, anc=None, lse=False):
    import torch
    from speculative_decoding_tree_ddtree_gb300 import lucetree as LT
    B, N, Hq, Hkv, D = cfg.B, cfg.N, cfg.Hq, cfg.Hkv, cfg.D
    dev = d["q"].device
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if anc is None:
        anc = torch.empty(B, N, dtype=torch.int64, device=dev)
        LT.lucetree_build_anc_mask(d["parent"], anc, status)
    ws = torch.empty(LT.lucetree_verify_attn_workspace(B, N, Hq, Hkv, D), dtype=torch.uint8, device=dev)
    ws.fill_(0x3F)  # finite garbage (0.747f): a partial read before it is written shows up as a wrong result
    out = torch.full((B, N, Hq, D), float("nan"), dtype=torch.float32, device=dev)
    lse_t = torch.full((B, N, Hq), float("nan"), dtype=torch.float32, device=dev) if lse else None
    LT.lucetree_verify_attn(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["ctx_len"], d["k_tree"],
                            d["v_tree"], anc, out, status, ws, lse=lse_t)
    torch.cuda.synchronize()
    return out, lse_t, int(status.item())
