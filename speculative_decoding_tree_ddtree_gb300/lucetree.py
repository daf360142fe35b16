"""Thin Python binding of liblucetree.so (include/lucetree.h).

Argument marshalling only: torch tensors become raw device pointers and every
step runs in the library's CUDA kernels.  The functions carry the C names.
There is no fallback: if the shared library is missing or a call returns an
error status, a ``LucetreeError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblucetree.so")

LUCETREE_OK = 0
LUCETREE_V_SAME, LUCETREE_V_INT8, LUCETREE_V_INT4 = 0, 1, 2
LUCETREE_K_SAME, LUCETREE_K_E4M3 = 0, 1
LUCETREE_F16 = 0
LUCETREE_BF16 = 1
PAGE_SIZE = 64
MAX_NODES = 64

DEV_BAD_PARENT = 0x1
DEV_BAD_PAGE = 0x2
DEV_BAD_CTX = 0x4
DEV_BAD_TOKEN = 0x8
DEV_BAD_NODE = 0x10
DEV_TIMEOUT = 0x20
DEV_NONFINITE = 0x40

EXPORTED = (
    "lucetree_verify_attn_workspace",
    "lucetree_verify_attn",
    "lucetree_build_anc_mask",
    "lucetree_argmax_workspace",
    "lucetree_argmax",
    "lucetree_accept",
    "lucetree_commit",
    "lucetree_status_string",
    "lucetree_abi_version",
    "lucetree_verify_attn_noalloc",
    "lucetree_lmhead_argmax_workspace",
    "lucetree_lmhead_argmax",
    "lucetree_delta_tree",
    "lucetree_delta_commit",
    "lucetree_stage_pages",
    "lucetree_verify_attn_vq",
    "lucetree_selftest_wait_timeout",
    "lucetree_verify_step_workspace",
    "lucetree_verify_step",
    "lucetree_verify_attn_kq_workspace",
    "lucetree_verify_attn_kq",
    "lucetree_commit_kq",
)


class LucetreeError(RuntimeError):
    pass


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int), ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hq", ctypes.c_int),
        ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("page_size", ctypes.c_int), ("scale", ctypes.c_float),
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("num_pages", ctypes.c_int), ("page_table", ctypes.c_void_p), ("max_pages_per_seq", ctypes.c_int),
        ("ctx_len", ctypes.c_void_p), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
        ("anc_mask", ctypes.c_void_p), ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


class StepArgs(ctypes.Structure):
    _fields_ = [
        ("attn", AttnArgs), ("parent", ctypes.c_void_p), ("draft", ctypes.c_void_p), ("logits", ctypes.c_void_p),
        ("vocab", ctypes.c_int), ("argmax", ctypes.c_void_p), ("acc_nodes", ctypes.c_void_p),
        ("acc_len", ctypes.c_void_p), ("bonus", ctypes.c_void_p), ("ctx_len_out", ctypes.c_void_p),
    ]


class CommitArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int), ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("page_size", ctypes.c_int), ("k_tree", ctypes.c_void_p), ("v_tree", ctypes.c_void_p),
        ("acc_nodes", ctypes.c_void_p), ("acc_len", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_int), ("num_pages", ctypes.c_int), ("ctx_len_in", ctypes.c_void_p),
        ("ctx_len_out", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


class LmHeadArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int), ("rows", ctypes.c_int), ("d_model", ctypes.c_int), ("vocab", ctypes.c_int),
        ("hidden", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("out_idx", ctypes.c_void_p),
        ("out_logit", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


class DeltaArgs(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int), ("B", ctypes.c_int), ("N", ctypes.c_int), ("Hk", ctypes.c_int),
        ("Hv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("parent", ctypes.c_void_p),
        ("state", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("acc_nodes", ctypes.c_void_p), ("acc_len", ctypes.c_void_p), ("status", ctypes.c_void_p),
    ]


class StageArgs(ctypes.Structure):
    _fields_ = [
        ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("n", ctypes.c_int),
        ("host_k", ctypes.c_void_p), ("host_v", ctypes.c_void_p), ("host_pages", ctypes.c_int),
        ("src", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("table_idx", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("table_len", ctypes.c_int),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("num_pages", ctypes.c_int),
        ("status", ctypes.c_void_p),
    ]


_lib = None


def load(path: str | None = None):
    """Load liblucetree.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise LucetreeError(f"{p} is missing: build it with speculative_decoding_tree_ddtree_gb300.build.build()")
    lib = ctypes.CDLL(p)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.lucetree_verify_attn_workspace.argtypes = [I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.lucetree_verify_attn.argtypes = [ctypes.POINTER(AttnArgs), P, SZ, P]
    lib.lucetree_build_anc_mask.argtypes = [P, I, I, P, P, P]
    lib.lucetree_argmax_workspace.argtypes = [I, I, ctypes.POINTER(SZ)]
    lib.lucetree_argmax.argtypes = [P, I, I, ctypes.c_longlong, P, P, SZ, P]
    lib.lucetree_accept.argtypes = [P, P, P, I, I, I, P, P, P, P, P]
    lib.lucetree_commit.argtypes = [ctypes.POINTER(CommitArgs), P]
    lib.lucetree_status_string.argtypes = [I]
    lib.lucetree_status_string.restype = ctypes.c_char_p
    lib.lucetree_abi_version.argtypes = []
    lib.lucetree_verify_attn_noalloc.argtypes = [ctypes.POINTER(AttnArgs), P]
    lib.lucetree_lmhead_argmax_workspace.argtypes = [I, ctypes.POINTER(SZ)]
    lib.lucetree_lmhead_argmax.argtypes = [ctypes.POINTER(LmHeadArgs), P, SZ, P]
    lib.lucetree_delta_tree.argtypes = [ctypes.POINTER(DeltaArgs), P]
    lib.lucetree_delta_commit.argtypes = [ctypes.POINTER(DeltaArgs), P]
    lib.lucetree_stage_pages.argtypes = [ctypes.POINTER(StageArgs), P]
    lib.lucetree_verify_attn_vq.argtypes = [ctypes.POINTER(AttnArgs), I, P, P, SZ, P]
    lib.lucetree_selftest_wait_timeout.argtypes = [P, ctypes.c_longlong, P, P]
    lib.lucetree_verify_step_workspace.argtypes = [I, I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.lucetree_verify_step.argtypes = [ctypes.POINTER(StepArgs), P, SZ, P]
    lib.lucetree_verify_attn_kq_workspace.argtypes = [I, I, I, I, I, ctypes.POINTER(SZ)]
    lib.lucetree_verify_attn_kq.argtypes = [ctypes.POINTER(AttnArgs), P, I, P, P, SZ, P]
    lib.lucetree_commit_kq.argtypes = [ctypes.POINTER(CommitArgs), P, P]
    for name in EXPORTED:
        if name not in ("lucetree_status_string", "lucetree_abi_version"):
            getattr(lib, name).restype = I
    if path is None:
        _lib = lib
    return lib


def _check(rc: int):
    if rc != LUCETREE_OK:
        msg = load().lucetree_status_string(rc).decode()
        raise LucetreeError(f"lucetree error {rc}: {msg}")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise LucetreeError("lucetree takes device tensors")
    if not t.is_contiguous():
        raise LucetreeError("lucetree takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# Element types the kernels read and write: 16-bit activations, int32 indices
# and lengths, fp32 outputs, 32-bit status words, 64-bit ancestor masks.
_H16 = (torch.float16, torch.bfloat16)
_I32 = (torch.int32,)
_F32 = (torch.float32,)
_W32 = tuple(t for t in (torch.int32, getattr(torch, "uint32", None)) if t is not None)
_W64 = tuple(t for t in (torch.int64, getattr(torch, "uint64", None)) if t is not None)
_U8 = (torch.uint8, torch.int8)


def _dims(t, name: str, ndim: int):
    """The shape of a required tensor of rank ndim."""
    if t is None:
        raise LucetreeError(f"{name} is required")
    if t.dim() != ndim:
        raise LucetreeError(f"{name}: expected {ndim} dimensions, got shape {tuple(t.shape)}")
    return t.shape


def _expect(t, name: str, shape: tuple, dtypes: tuple):
    """Refuse a tensor whose shape or element type differs from what the
    kernel will index: a mismatch would read or write past its end."""
    if t is None:
        raise LucetreeError(f"{name} is required")
    if t.dtype in dtypes and t.shape == shape:
        return
    raise LucetreeError(f"{name}: expected shape {tuple(shape)} of {'/'.join(str(d) for d in dtypes)}, "
                        f"got {tuple(t.shape)} of {t.dtype}")


def _expect_status(t):
    if t is None or t.dtype not in _W32 or t.numel() < 1:
        raise LucetreeError("status: expected a device int32 word")


def _expect_16bit(t, name: str, shape: tuple):
    """Raw 16-bit data of any 16-bit element type (byte copies)."""
    if t is None:
        raise LucetreeError(f"{name} is required")
    if t.element_size() != 2 or t.shape != shape:
        raise LucetreeError(f"{name}: expected shape {tuple(shape)} of a 16-bit type, got {tuple(t.shape)} of {t.dtype}")


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LUCETREE_BF16
    if t.dtype == torch.float16:
        return LUCETREE_F16
    raise LucetreeError(f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------- entry points

def lucetree_verify_attn_workspace(B: int, N: int, Hq: int, Hkv: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lucetree_verify_attn_workspace(B, N, Hq, Hkv, D, ctypes.byref(n)))
    return int(n.value)


def _check_attn(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse,
                v_format=None, v_exp=None, k_exp=None):
    """Shapes and element types of one tree-verify attention call (layouts as
    lucetree_verify_attn documents them); v_format selects the quantised V
    pool, k_exp the E4M3 K pool (k_pool then holds the codes)."""
    B, N, Hq, D = _dims(q, "q", 4)
    if q.dtype not in _H16:
        raise LucetreeError(f"q: unsupported dtype {q.dtype}")
    P, Hkv, page, _ = _dims(k_pool, "k_pool", 4)
    if k_exp is None:
        _expect(k_pool, "k_pool", (P, Hkv, page, D), (q.dtype,))
    else:
        _expect(k_pool, "k_codes", (P, Hkv, page, D), _U8)
        _expect(k_exp, "k_exp", (P, Hkv, page), _U8)
    if v_format is None or v_format == LUCETREE_V_SAME:
        _expect(v_pool, "v_pool", (P, Hkv, page, D), (q.dtype,))
    else:
        _expect(v_pool, "v_codes", (P, Hkv, page, D // 2 if v_format == LUCETREE_V_INT4 else D), _U8)
        _expect(v_exp, "v_exp", (P, Hkv, page), _U8)
    _expect(k_tree, "k_tree", (B, N, Hkv, D), (q.dtype,))
    _expect(v_tree, "v_tree", (B, N, Hkv, D), (q.dtype,))
    _expect(page_table, "page_table", (B, _dims(page_table, "page_table", 2)[1]), _I32)
    _expect(ctx_len, "ctx_len", (B,), _I32)
    _expect(anc_mask, "anc_mask", (B, N), _W64)
    _expect(out, "out", (B, N, Hq, D), _F32)
    if lse is not None:
        _expect(lse, "lse", (B, N, Hq), _F32)
    _expect_status(status)


def _attn_args(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, scale,
               v_format=None, v_exp=None, k_exp=None):
    _check_attn(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, v_format, v_exp,
                k_exp)
    B, N, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    a = AttnArgs()
    a.dtype = dtype_code(q)
    a.B, a.N, a.Hq, a.Hkv, a.D = B, N, Hq, Hkv, D
    a.page_size = k_pool.shape[2]
    a.scale = float(scale) if scale is not None else float(D) ** -0.5
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.num_pages = k_pool.shape[0]
    a.page_table, a.max_pages_per_seq = _ptr(page_table), page_table.shape[1]
    a.ctx_len, a.k_tree, a.v_tree, a.anc_mask = _ptr(ctx_len), _ptr(k_tree), _ptr(v_tree), _ptr(anc_mask)
    a.out, a.lse, a.status = _ptr(out), _ptr(lse), _ptr(status)
    return a


def lucetree_verify_attn(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status,
                         workspace, lse=None, scale: float | None = None, stream=None):
    """q [B][N][Hq][D]; pools [P][Hkv][64][D]; page_table int32 [B][max_pages];
    ctx_len int32 [B]; tree K/V [B][N][Hkv][D]; anc_mask int64 [B][N];
    out fp32 [B][N][Hq][D]; status int32 [1]; workspace uint8 (see
    lucetree_verify_attn_workspace)."""
    a = _attn_args(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, scale)
    _check(load().lucetree_verify_attn(ctypes.byref(a), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))



def lucetree_verify_attn_vq(q, k_pool, v_codes, v_exp, v_format, page_table, ctx_len, k_tree, v_tree, anc_mask, out,
                            status, workspace, lse=None, scale: float | None = None, stream=None):
    """As lucetree_verify_attn with V stored quantised: v_codes uint8 [P][Hkv][64][D]
    (int8 codes) or [P][Hkv][64][D/2] (int4 codes, low nibble first), v_exp uint8
    [P][Hkv][64] (value = code * 2^(e - 127))."""
    if v_format not in (LUCETREE_V_INT8, LUCETREE_V_INT4):
        raise LucetreeError(f"unsupported V format {v_format}")
    a = _attn_args(q, k_pool, v_codes, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, scale,
                   v_format=v_format, v_exp=v_exp)
    _check(load().lucetree_verify_attn_vq(ctypes.byref(a), int(v_format), _ptr(v_exp), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def lucetree_verify_attn_kq_workspace(B: int, N: int, Hq: int, Hkv: int, D: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lucetree_verify_attn_kq_workspace(B, N, Hq, Hkv, D, ctypes.byref(n)))
    return int(n.value)


def lucetree_verify_attn_kq(q, k_codes, k_exp, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status,
                            workspace, v_format=LUCETREE_V_SAME, v_exp=None, lse=None, scale: float | None = None,
                            stream=None):
    """As lucetree_verify_attn with K stored as FP8 E4M3: k_codes uint8
    [P][Hkv][64][D], k_exp uint8 [P][Hkv][64] (value = e4m3(code) * 2^(e - 127));
    V in q's dtype (v_format LUCETREE_V_SAME) or as int8 / int4 codes with
    v_exp.  bf16 queries, D = 256; workspace from lucetree_verify_attn_kq_workspace."""
    if v_format not in (LUCETREE_V_SAME, LUCETREE_V_INT8, LUCETREE_V_INT4):
        raise LucetreeError(f"unsupported V format {v_format}")
    a = _attn_args(q, k_codes, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, scale,
                   v_format=v_format, v_exp=v_exp, k_exp=k_exp)
    _check(load().lucetree_verify_attn_kq(ctypes.byref(a), _ptr(k_exp), int(v_format), _ptr(v_exp), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def lucetree_build_anc_mask(parent, anc, status, stream=None):
    B, N = _dims(parent, "parent", 2)
    _expect(parent, "parent", (B, N), _I32)
    _expect(anc, "anc", (B, N), _W64)
    _expect_status(status)
    _check(load().lucetree_build_anc_mask(_ptr(parent), B, N, _ptr(anc), _ptr(status), _stream(stream)))


def lucetree_argmax_workspace(rows: int, vocab: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lucetree_argmax_workspace(rows, vocab, ctypes.byref(n)))
    return int(n.value)


def lucetree_argmax(logits, out_idx, workspace, stream=None):
    """logits fp32 [..., V] (rows = all leading dims) -> out_idx int32 [...]."""
    if logits is None or logits.dim() < 1 or logits.dtype != torch.float32:
        raise LucetreeError("logits: expected a float32 tensor [..., V]")
    V = logits.shape[-1]
    rows = logits.numel() // V if V > 0 else 0
    if out_idx is None or out_idx.dtype != torch.int32 or out_idx.numel() != rows:
        raise LucetreeError(f"out_idx: expected {rows} int32 entries")
    _check(load().lucetree_argmax(_ptr(logits), rows, V, V, _ptr(out_idx), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def lucetree_accept(parent, draft, argmax_idx, vocab: int, acc_nodes, acc_len, bonus, status, stream=None):
    B, N = _dims(parent, "parent", 2)
    _expect(parent, "parent", (B, N), _I32)
    _expect(draft, "draft", (B, N), _I32)
    _expect(argmax_idx, "argmax", (B, N + 1), _I32)
    _expect(acc_nodes, "acc_nodes", (B, N), _I32)
    _expect(acc_len, "acc_len", (B,), _I32)
    _expect(bonus, "bonus", (B,), _I32)
    _expect_status(status)
    _check(load().lucetree_accept(_ptr(parent), _ptr(draft), _ptr(argmax_idx), B, N, vocab, _ptr(acc_nodes),
                                  _ptr(acc_len), _ptr(bonus), _ptr(status), _stream(stream)))


def lucetree_commit(k_tree, v_tree, acc_nodes, acc_len, page_table, ctx_len_in, ctx_len_out, k_pool, v_pool,
                    status, stream=None):
    B, N, Hkv, D = _dims(k_tree, "k_tree", 4)
    if k_tree.dtype not in _H16:
        raise LucetreeError(f"k_tree: unsupported dtype {k_tree.dtype}")
    _expect(v_tree, "v_tree", (B, N, Hkv, D), (k_tree.dtype,))
    _expect(acc_nodes, "acc_nodes", (B, N), _I32)
    _expect(acc_len, "acc_len", (B,), _I32)
    _expect(page_table, "page_table", (B, _dims(page_table, "page_table", 2)[1]), _I32)
    _expect(ctx_len_in, "ctx_len_in", (B,), _I32)
    _expect(ctx_len_out, "ctx_len_out", (B,), _I32)
    P, _, page, _ = _dims(k_pool, "k_pool", 4)
    _expect(k_pool, "k_pool", (P, Hkv, page, D), (k_tree.dtype,))
    _expect(v_pool, "v_pool", (P, Hkv, page, D), (k_tree.dtype,))
    _expect_status(status)
    c = CommitArgs()
    c.dtype = dtype_code(k_tree)
    c.B, c.N, c.Hkv, c.D = B, N, Hkv, D
    c.page_size = k_pool.shape[2]
    c.k_tree, c.v_tree = _ptr(k_tree), _ptr(v_tree)
    c.acc_nodes, c.acc_len = _ptr(acc_nodes), _ptr(acc_len)
    c.page_table, c.max_pages_per_seq = _ptr(page_table), page_table.shape[1]
    c.num_pages = k_pool.shape[0]
    c.ctx_len_in, c.ctx_len_out = _ptr(ctx_len_in), _ptr(ctx_len_out)
    c.k_pool, c.v_pool, c.status = _ptr(k_pool), _ptr(v_pool), _ptr(status)
    _check(load().lucetree_commit(ctypes.byref(c), _stream(stream)))


def lucetree_commit_kq(k_tree, v_tree, acc_nodes, acc_len, page_table, ctx_len_in, ctx_len_out, k_codes, k_exp,
                       v_pool, status, stream=None):
    """lucetree_commit into a K pool held as E4M3 codes (k_codes uint8
    [P][Hkv][64][D], k_exp uint8 [P][Hkv][64]): each accepted K row is stored
    quantised; V rows are copied into the bf16 v_pool."""
    B, N, Hkv, D = _dims(k_tree, "k_tree", 4)
    if k_tree.dtype != torch.bfloat16:
        raise LucetreeError(f"k_tree: expected bfloat16, got {k_tree.dtype}")
    _expect(v_tree, "v_tree", (B, N, Hkv, D), (k_tree.dtype,))
    _expect(acc_nodes, "acc_nodes", (B, N), _I32)
    _expect(acc_len, "acc_len", (B,), _I32)
    _expect(page_table, "page_table", (B, _dims(page_table, "page_table", 2)[1]), _I32)
    _expect(ctx_len_in, "ctx_len_in", (B,), _I32)
    _expect(ctx_len_out, "ctx_len_out", (B,), _I32)
    P, _, page, _ = _dims(k_codes, "k_codes", 4)
    _expect(k_codes, "k_codes", (P, Hkv, page, D), _U8)
    _expect(k_exp, "k_exp", (P, Hkv, page), _U8)
    _expect(v_pool, "v_pool", (P, Hkv, page, D), (k_tree.dtype,))
    _expect_status(status)
    c = CommitArgs()
    c.dtype = dtype_code(k_tree)
    c.B, c.N, c.Hkv, c.D = B, N, Hkv, D
    c.page_size = page
    c.k_tree, c.v_tree = _ptr(k_tree), _ptr(v_tree)
    c.acc_nodes, c.acc_len = _ptr(acc_nodes), _ptr(acc_len)
    c.page_table, c.max_pages_per_seq = _ptr(page_table), page_table.shape[1]
    c.num_pages = P
    c.ctx_len_in, c.ctx_len_out = _ptr(ctx_len_in), _ptr(ctx_len_out)
    c.k_pool, c.v_pool, c.status = _ptr(k_codes), _ptr(v_pool), _ptr(status)
    _check(load().lucetree_commit_kq(ctypes.byref(c), _ptr(k_exp), _stream(stream)))


# ---------------------------------------------------------------- one whole step

def lucetree_verify_step_workspace(B: int, N: int, Hq: int, Hkv: int, D: int, vocab: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lucetree_verify_step_workspace(B, N, Hq, Hkv, D, vocab, ctypes.byref(n)))
    return int(n.value)


def _step_args(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, parent, draft, logits, out, lse, argmax_idx,
               acc_nodes, acc_len, bonus, ctx_len_out, status, scale=None):
    """Checks every tensor of one fused step against the documented layouts and
    packs the C argument struct."""
    B, N, Hq, D = _dims(q, "q", 4)
    _expect(parent, "parent", (B, N), _I32)
    _expect(draft, "draft", (B, N), _I32)
    V = _dims(logits, "logits", 3)[2]
    _expect(logits, "logits", (B, N + 1, V), _F32)
    _expect(argmax_idx, "argmax", (B, N + 1), _I32)
    _expect(acc_nodes, "acc_nodes", (B, N), _I32)
    _expect(acc_len, "acc_len", (B,), _I32)
    _expect(bonus, "bonus", (B,), _I32)
    _expect(ctx_len_out, "ctx_len_out", (B,), _I32)
    if ctx_len_out.data_ptr() == ctx_len.data_ptr():
        raise LucetreeError("ctx_len_out must not alias ctx_len in the fused step")
    anc_dummy = torch.empty((B, N), dtype=torch.int64, device="meta")
    _check_attn(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_dummy, out, status, lse)
    s = StepArgs()
    a = s.attn
    a.dtype = dtype_code(q)
    a.B, a.N, a.Hq, a.Hkv, a.D = B, N, Hq, k_pool.shape[1], D
    a.page_size = k_pool.shape[2]
    a.scale = float(scale) if scale is not None else float(D) ** -0.5
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.num_pages = k_pool.shape[0]
    a.page_table, a.max_pages_per_seq = _ptr(page_table), page_table.shape[1]
    a.ctx_len, a.k_tree, a.v_tree, a.anc_mask = _ptr(ctx_len), _ptr(k_tree), _ptr(v_tree), None
    a.out, a.lse, a.status = _ptr(out), _ptr(lse), _ptr(status)
    s.parent, s.draft, s.logits, s.vocab = _ptr(parent), _ptr(draft), _ptr(logits), V
    s.argmax, s.acc_nodes, s.acc_len, s.bonus = _ptr(argmax_idx), _ptr(acc_nodes), _ptr(acc_len), _ptr(bonus)
    s.ctx_len_out = _ptr(ctx_len_out)
    return s


class VerifyStep:
    """Device buffers and workspaces for repeated verify steps of one shape.

    ``run`` issues the whole step (ancestor masks, tree-verify attention,
    argmax, acceptance and commit, all library kernels) as ONE C call,
    lucetree_verify_step.  The tensors of a call are checked against the
    documented layouts the first time that set of buffers is seen; later
    calls with the same buffers reuse the packed arguments, so a step costs
    one ctypes call on the host."""

    def __init__(self, B, N, Hq, Hkv, D, vocab, device="cuda"):
        self.B, self.N, self.Hq, self.Hkv, self.D, self.vocab = B, N, Hq, Hkv, D, vocab
        dev = torch.device(device)
        # zeroed once: the step's counters must start at zero and every call leaves them so
        self.ws_step = torch.zeros(lucetree_verify_step_workspace(B, N, Hq, Hkv, D, vocab), dtype=torch.uint8,
                                   device=dev)
        self.ws_attn = torch.empty(lucetree_verify_attn_workspace(B, N, Hq, Hkv, D), dtype=torch.uint8, device=dev)
        self.ws_argmax = torch.empty(lucetree_argmax_workspace(B * (N + 1), vocab), dtype=torch.uint8, device=dev)
        self.anc = torch.empty(B, N, dtype=torch.int64, device=dev)
        self.out = torch.empty(B, N, Hq, D, dtype=torch.float32, device=dev)
        self.lse = torch.empty(B, N, Hq, dtype=torch.float32, device=dev)
        self.argmax = torch.empty(B, N + 1, dtype=torch.int32, device=dev)
        # the step's result in one contiguous int32 buffer (one copy reads it
        # back): accepted path [B][N], accepted count [B], bonus token [B],
        # new committed length [B]
        self.results = torch.empty(B * N + 3 * B, dtype=torch.int32, device=dev)
        self.acc_nodes = self.results[:B * N].view(B, N)
        self.acc_len = self.results[B * N:B * N + B]
        self.bonus = self.results[B * N + B:B * N + 2 * B]
        self.ctx_out = self.results[B * N + 2 * B:]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._packed = {}

    def run(self, q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, parent, draft, logits, stream=None):
        ts = (q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, parent, draft, logits)
        key = tuple((t.data_ptr(), tuple(t.shape), t.dtype, t.is_contiguous()) for t in ts)
        s = self._packed.get(key)
        if s is None:
            s = _step_args(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, parent, draft, logits, self.out,
                           self.lse, self.argmax, self.acc_nodes, self.acc_len, self.bonus, self.ctx_out, self.status)
            if len(self._packed) > 64:
                self._packed.clear()
            self._packed[key] = s
        _check(load().lucetree_verify_step(ctypes.byref(s), _ptr(self.ws_step), self.ws_step.numel(),
                                           _stream(stream)))

    def run_calls(self, q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, parent, draft, logits, stream=None):
        """The same step as the five separate C calls (masks, attention,
        argmax, acceptance, commit)."""
        lucetree_build_anc_mask(parent, self.anc, self.status, stream)
        lucetree_verify_attn(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, self.anc, self.out,
                             self.status, self.ws_attn, lse=self.lse, stream=stream)
        lucetree_argmax(logits, self.argmax, self.ws_argmax, stream)
        lucetree_accept(parent, draft, self.argmax, self.vocab, self.acc_nodes, self.acc_len, self.bonus,
                        self.status, stream)
        lucetree_commit(k_tree, v_tree, self.acc_nodes, self.acc_len, page_table, ctx_len, self.ctx_out, k_pool,
                        v_pool, self.status, stream)


# ---------------------------------------------------------------- allocation-free variant

NOALLOC_SCRATCH_BYTES = 32 << 20  # LUCETREE_NOALLOC_SCRATCH_BYTES of include/lucetree.h


def lucetree_verify_attn_noalloc(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status,
                                 lse=None, scale: float | None = None, stream=None):
    """lucetree_verify_attn for callers that cannot allocate device memory: the
    split-K scratch is a fixed 32 MiB device array inside the library (shared
    by every call on a device; calls that overlap on the GPU race on it).  The
    first call in a context may load the library's device code to find that
    array, so make it before any stream capture.  Shapes whose workspace
    would exceed 32 MiB raise."""
    B, N, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    need = lucetree_verify_attn_workspace(B, N, Hq, Hkv, D)
    if need > NOALLOC_SCRATCH_BYTES:
        raise LucetreeError(f"lucetree_verify_attn_noalloc: these sizes need {need} bytes of scratch, "
                            f"more than the fixed {NOALLOC_SCRATCH_BYTES}")
    a = _attn_args(q, k_pool, v_pool, page_table, ctx_len, k_tree, v_tree, anc_mask, out, status, lse, scale)
    _check(load().lucetree_verify_attn_noalloc(ctypes.byref(a), _stream(stream)))


# ---------------------------------------------------------------- lm_head projection + argmax

def lucetree_lmhead_argmax_workspace(rows: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().lucetree_lmhead_argmax_workspace(rows, ctypes.byref(n)))
    return int(n.value)


def lucetree_lmhead_argmax(hidden, weight, out_idx, status, workspace, out_logit=None, stream=None):
    """hidden [rows][d_model] and weight [vocab][d_model] (both fp16 or both
    bf16) -> out_idx int32 [rows]: the lowest vocabulary index of each row's
    largest logit; optionally out_logit fp32 [rows] (that logit)."""
    rows, d_model = _dims(hidden, "hidden", 2)
    a = LmHeadArgs()
    a.dtype = dtype_code(hidden)
    _expect(weight, "weight", (_dims(weight, "weight", 2)[0], d_model), (hidden.dtype,))
    _expect(out_idx, "out_idx", (rows,), _I32)
    if out_logit is not None:
        _expect(out_logit, "out_logit", (rows,), _F32)
    _expect_status(status)
    a.rows, a.d_model, a.vocab = rows, d_model, weight.shape[0]
    a.hidden, a.weight = _ptr(hidden), _ptr(weight)
    a.out_idx, a.out_logit, a.status = _ptr(out_idx), _ptr(out_logit), _ptr(status)
    _check(load().lucetree_lmhead_argmax(ctypes.byref(a), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))


# ---------------------------------------------------------------- recurrent-state (delta rule) step

def _delta_args(q, k, v, alpha, beta, state, status, parent=None, out=None, acc_nodes=None, acc_len=None,
                tree=True):
    B, N, Hk, dk = _dims(k, "k", 4)
    Hv, dv = _dims(v, "v", 4)[2:]
    a = DeltaArgs()
    a.dtype = dtype_code(k)
    _expect(v, "v", (B, N, Hv, dv), (k.dtype,))
    _expect(alpha, "alpha", (B, N, Hv), _F32)
    _expect(beta, "beta", (B, N, Hv), _F32)
    _expect(state, "state", (B, Hv, dk, dv), _F32)
    _expect_status(status)
    if tree:
        _expect(q, "q", (B, N, Hk, dk), (k.dtype,))
        _expect(parent, "parent", (B, N), _I32)
        _expect(out, "out", (B, N, Hv, dv), _F32)
    else:
        _expect(acc_nodes, "acc_nodes", (B, N), _I32)
        _expect(acc_len, "acc_len", (B,), _I32)
    a.B, a.N, a.Hk, a.Hv, a.dk, a.dv = B, N, Hk, Hv, dk, dv
    a.q, a.k, a.v = _ptr(q), _ptr(k), _ptr(v)
    a.alpha, a.beta, a.parent = _ptr(alpha), _ptr(beta), _ptr(parent)
    a.state, a.out, a.status = _ptr(state), _ptr(out), _ptr(status)
    a.acc_nodes, a.acc_len = _ptr(acc_nodes), _ptr(acc_len)
    return a


def lucetree_delta_tree(q, k, v, alpha, beta, parent, state, out, status, stream=None):
    """out[b][i][h] = S_i^T q_i with S_i the gated-delta-rule state along node
    i's root path from state[b][h] (fp32); the state is only read."""
    a = _delta_args(q, k, v, alpha, beta, state, status, parent=parent, out=out)
    _check(load().lucetree_delta_tree(ctypes.byref(a), _stream(stream)))


def lucetree_delta_commit(k, v, alpha, beta, acc_nodes, acc_len, state, status, stream=None):
    """state[b][h] <- the recurrence along acc_nodes[b][:acc_len[b]] (in place)."""
    a = _delta_args(None, k, v, alpha, beta, state, status, acc_nodes=acc_nodes, acc_len=acc_len, tree=False)
    _check(load().lucetree_delta_commit(ctypes.byref(a), _stream(stream)))


# ---------------------------------------------------------------- host-resident pages

def _host_ptr(t: torch.Tensor) -> ctypes.c_void_p:
    if t.is_cuda or not t.is_pinned():
        raise LucetreeError("host pools must be page-locked host tensors")
    if not t.is_contiguous():
        raise LucetreeError("lucetree takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def lucetree_stage_pages(host_k, host_v, src, dst, k_pool, v_pool, status, table_idx=None, page_table=None,
                         stream=None):
    """Copy host pages src[i] (page-locked host pools [host_pages][Hkv][64][D])
    into device pool pages dst[i]; with table_idx, page_table.view(-1)[table_idx[i]] = dst[i]."""
    P, Hkv, page, D = _dims(k_pool, "k_pool", 4)
    _expect_16bit(k_pool, "k_pool", (P, Hkv, page, D))
    _expect_16bit(v_pool, "v_pool", (P, Hkv, page, D))
    host_pages = _dims(host_k, "host_k", 4)[0]
    _expect_16bit(host_k, "host_k", (host_pages, Hkv, page, D))
    _expect_16bit(host_v, "host_v", (host_pages, Hkv, page, D))
    n = _dims(src, "src", 1)[0]
    _expect(src, "src", (n,), _I32)
    _expect(dst, "dst", (n,), _I32)
    if table_idx is not None:
        _expect(table_idx, "table_idx", (n,), _I32)
        if page_table is None or page_table.dtype != torch.int32:
            raise LucetreeError("page_table: an int32 table is required with table_idx")
    _expect_status(status)
    a = StageArgs()
    a.Hkv, a.D = k_pool.shape[1], k_pool.shape[3]
    a.n = src.numel()
    a.host_k, a.host_v, a.host_pages = _host_ptr(host_k), _host_ptr(host_v), host_k.shape[0]
    a.src, a.dst, a.table_idx = _ptr(src), _ptr(dst), _ptr(table_idx)
    a.page_table = _ptr(page_table)
    a.table_len = page_table.numel() if page_table is not None else 0
    a.k_pool, a.v_pool, a.num_pages = _ptr(k_pool), _ptr(v_pool), k_pool.shape[0]
    a.status = _ptr(status)
    _check(load().lucetree_stage_pages(ctypes.byref(a), _stream(stream)))


# ---------------------------------------------------------------- failure path self-test

def lucetree_selftest_wait_timeout(status, limit_cycles: int, waited_cycles=None, stream=None):
    """One block waits on a barrier nothing arrives on; after ~limit_cycles SM
    cycles it sets DEV_TIMEOUT in status and returns (waited_cycles: int64 [1])."""
    _expect_status(status)
    if waited_cycles is not None:
        _expect(waited_cycles, "waited_cycles", (1,), (torch.int64,))
    _check(load().lucetree_selftest_wait_timeout(_ptr(status), int(limit_cycles), _ptr(waited_cycles),
                                                 _stream(stream)))
