"""fp64 CPU oracle for the DDTree verify step -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It shares nothing with the CUDA path.
The arithmetic lives in ``lucetree_oracle.c`` (plain C, fp64); this module
builds it with gcc and marshals numpy arrays.  Every function below states the
rule it follows; the C file carries the citations and the pins are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lucetree_oracle.c")
_LIB = os.path.join(_HERE, "liblucetree_oracle.so")
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags only)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_verify_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, f64, P, P, P, i32, P, i32,
                                           P, P, P, P, P, i64, P, P, i32]
        lib.oracle_verify_attn.restype = i32
        lib.oracle_argmax.argtypes = [P, i64, i64, i64, P]
        lib.oracle_argmax.restype = None
        lib.oracle_accept.argtypes = [i32, i32, P, P, P, P, P, P]
        lib.oracle_accept.restype = i32
        lib.oracle_commit.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, i32, i32, P, P, P]
        lib.oracle_commit.restype = i32
        lib.oracle_ancestor_matrix.argtypes = [P, i32, P]
        lib.oracle_ancestor_matrix.restype = None
        lib.oracle_upcast.argtypes = [i32, ctypes.c_uint16]
        lib.oracle_lmhead_argmax.argtypes = [i32, i64, i64, i64, P, P, P, P, P, i32]
        lib.oracle_lmhead_argmax.restype = i32
        lib.oracle_upcast.restype = f64
        lib.oracle_delta_tree.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.oracle_delta_tree.restype = i32
        lib.oracle_delta_commit.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P]
        lib.oracle_delta_commit.restype = i32
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def upcast(dtype: int, bits: int) -> float:
    """Exact value of one fp16 (dtype 0) or bf16 (dtype 1) bit pattern."""
    return _load().oracle_upcast(dtype, bits)


def ancestor_matrix(parent) -> np.ndarray:
    """uint8 [N][N]: 1 iff node j is node i or an ancestor of i."""
    parent = _c(parent, np.int32)
    n = parent.shape[0]
    out = np.zeros((n, n), dtype=np.uint8)
    _load().oracle_ancestor_matrix(_p(parent), n, _p(out))
    return out


def verify_attn(inp: dict, dtype: int, scale: float | None = None, rows=None, threads: int | None = None):
    """Tree-verify attention in fp64 with an explicit mask.

    ``inp`` holds the generator's arrays.  ``rows`` (flat ids (b*N+i)*Hq+h)
    selects a subset; default all rows.  Returns (out [rows][D] fp64,
    lse [rows] natural log)."""
    q = _c(inp["q"], np.uint16)
    B, N, Hq, D = q.shape
    k_pool = _c(inp["k_pool"], np.uint16)
    v_pool = _c(inp["v_pool"], np.uint16)
    num_pages, Hkv, P, _ = k_pool.shape
    pt = _c(inp["page_table"], np.int32)
    ctx = _c(inp["ctx_len"], np.int32)
    kt = _c(inp["k_tree"], np.uint16)
    vt = _c(inp["v_tree"], np.uint16)
    par = _c(inp["parent"], np.int32)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if rows is None:
        rows_arr = None
        n_rows = B * N * Hq
    else:
        rows_arr = _c(rows, np.int32)
        n_rows = rows_arr.shape[0]
    out = np.zeros((n_rows, D), dtype=np.float64)
    lse = np.zeros(n_rows, dtype=np.float64)
    if threads is None:
        threads = os.cpu_count() or 1
    rc = _load().oracle_verify_attn(dtype, B, N, Hq, Hkv, D, P, float(scale), _p(q), _p(k_pool), _p(v_pool),
                                    num_pages, _p(pt), pt.shape[1], _p(ctx), _p(kt), _p(vt), _p(par),
                                    None if rows_arr is None else _p(rows_arr), n_rows, _p(out), _p(lse),
                                    int(threads))
    if rc != 0:
        raise ValueError(f"oracle_verify_attn failed ({rc})")
    return out, lse


def argmax(logits) -> np.ndarray:
    """First index of the maximum of each row of a 2-D float32 array."""
    x = _c(logits, np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty(x2.shape[0], dtype=np.int32)
    _load().oracle_argmax(_p(x2), x2.shape[0], x2.shape[1], x2.shape[1], _p(out))
    return out.reshape(x.shape[:-1])


def accept(parent, draft, argmax_idx):
    """Greedy acceptance; returns (acc_nodes [B][N] (-1 padded), acc_len [B], bonus [B])."""
    par = _c(parent, np.int32)
    dr = _c(draft, np.int32)
    am = _c(argmax_idx, np.int32)
    B, N = par.shape
    acc = np.full((B, N), -1, dtype=np.int32)
    alen = np.zeros(B, dtype=np.int32)
    bonus = np.zeros(B, dtype=np.int32)
    rc = _load().oracle_accept(B, N, _p(par), _p(dr), _p(am), _p(acc), _p(alen), _p(bonus))
    if rc != 0:
        raise ValueError("parent array is not in topological order")
    return acc, alen, bonus


def commit(inp: dict, acc_nodes, acc_len, inplace: bool = False):
    """Returns (k_pool, v_pool, ctx_len) after committing, on copies (or, with
    ``inplace``, writing into the given pools; ctx_len is always a copy)."""
    if inplace:
        k_pool, v_pool = inp["k_pool"], inp["v_pool"]
        assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous and k_pool.dtype == np.uint16
    else:
        k_pool = np.array(inp["k_pool"], dtype=np.uint16, copy=True)
        v_pool = np.array(inp["v_pool"], dtype=np.uint16, copy=True)
    ctx = np.array(inp["ctx_len"], dtype=np.int32, copy=True)
    kt = _c(inp["k_tree"], np.uint16)
    vt = _c(inp["v_tree"], np.uint16)
    pt = _c(inp["page_table"], np.int32)
    acc = _c(acc_nodes, np.int32)
    alen = _c(acc_len, np.int32)
    B, N, Hkv, D = kt.shape
    rc = _load().oracle_commit(B, N, Hkv, D, k_pool.shape[2], _p(kt), _p(vt), _p(acc), _p(alen), _p(pt),
                               pt.shape[1], k_pool.shape[0], _p(ctx), _p(k_pool), _p(v_pool))
    if rc != 0:
        raise ValueError("commit touched a page outside the pool")
    return k_pool, v_pool, ctx


def lmhead_argmax(hidden_bits, weight_bits, dtype: int, threads: int | None = None):
    """argmax_v of sum_d hidden[r][d] * weight[v][d] in fp64 (lowest index on
    ties), with each row's largest and second-largest logit.  hidden_bits
    [rows][d_model] and weight_bits [vocab][d_model] are uint16 storage bits."""
    h = _c(hidden_bits, np.uint16)
    w = _c(weight_bits, np.uint16)
    rows, d_model = h.shape
    vocab = w.shape[0]
    assert w.shape[1] == d_model
    out = np.empty(rows, np.int32)
    top1 = np.empty(rows, np.float64)
    top2 = np.empty(rows, np.float64)
    nt = threads or os.cpu_count() or 1
    rc = _load().oracle_lmhead_argmax(dtype, rows, d_model, vocab, _p(h), _p(w), _p(out), _p(top1), _p(top2), nt)
    if rc != 0:
        raise RuntimeError("oracle_lmhead_argmax failed")
    return out, top1, top2


def _delta_dims(inp: dict):
    B, N, Hk, dk = inp["q"].shape
    Hv, dv = inp["v"].shape[2], inp["v"].shape[3]
    return B, N, Hk, Hv, dk, dv


def delta_tree(inp: dict, dtype: int) -> np.ndarray:
    """Gated delta rule along each node's root path from the committed state:
    S_i = alpha_i (I - beta_i k_i k_i^T) S_parent + beta_i k_i v_i^T, o_i = S_i^T q_i.
    inp: q, k [B][N][Hk][dk] and v [B][N][Hv][dv] (uint16 bits), alpha, beta
    [B][N][Hv] float32, parent [B][N] int32, state [B][Hv][dk][dv] float32.
    Returns out [B][N][Hv][dv] float64."""
    B, N, Hk, Hv, dk, dv = _delta_dims(inp)
    q, k, v = (_c(inp[x], np.uint16) for x in ("q", "k", "v"))
    al, be = _c(inp["alpha"], np.float32), _c(inp["beta"], np.float32)
    par, st = _c(inp["parent"], np.int32), _c(inp["state"], np.float32)
    out = np.empty((B, N, Hv, dv), np.float64)
    rc = _load().oracle_delta_tree(dtype, B, N, Hk, Hv, dk, dv, _p(q), _p(k), _p(v), _p(al), _p(be), _p(par),
                                   _p(st), _p(out))
    if rc != 0:
        raise ValueError("oracle_delta_tree: bad parent array or sizes")
    return out


def delta_commit(inp: dict, dtype: int, acc_nodes, acc_len) -> np.ndarray:
    """The committed state after the recurrence along acc_nodes[b][:acc_len[b]]
    (root-to-leaf order) from inp["state"]: [B][Hv][dk][dv] float64."""
    B, N, Hk, Hv, dk, dv = _delta_dims(inp)
    k, v = _c(inp["k"], np.uint16), _c(inp["v"], np.uint16)
    al, be = _c(inp["alpha"], np.float32), _c(inp["beta"], np.float32)
    an, ln = _c(acc_nodes, np.int32), _c(acc_len, np.int32)
    st = _c(inp["state"], np.float32)
    out = np.empty((B, Hv, dk, dv), np.float64)
    rc = _load().oracle_delta_commit(dtype, B, N, Hk, Hv, dk, dv, _p(k), _p(v), _p(al), _p(be), _p(an), _p(ln),
                                     _p(st), _p(out))
    if rc != 0:
        raise ValueError("oracle_delta_commit: bad accepted path or sizes")
    return out


def stage_pages(host_k, host_v, src, dst, k_pool, v_pool, table_idx=None, page_table=None):
    """Host-resident KV pages brought back into the device pool.  The pages
    keep cold 64-token chunks in host memory ("Lucebox Hub", section
    "KVFlash"); bringing page src[i] back means pool[dst[i]] = host[src[i]]
    for K and V, and page_table.flat[table_idx[i]] = dst[i] when a table is
    given.  Returns new (k_pool, v_pool, page_table) arrays; inputs untouched."""
    kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    for s_, d_ in zip(np.asarray(src).tolist(), np.asarray(dst).tolist()):
        kp[d_] = host_k[s_]
        vp[d_] = host_v[s_]
    pt = None
    if page_table is not None:
        pt = np.array(page_table, copy=True)
        flat = pt.reshape(-1)
        for t, d_ in zip(np.asarray(table_idx).tolist(), np.asarray(dst).tolist()):
            flat[t] = d_
    return kp, vp, pt


V_INT8, V_INT4 = 1, 2


def dequant_v(codes, v_exp, v_format: int, dtype: int) -> np.ndarray:
    """Quantised V of the asymmetric K/V storage (the pages list K/V
    quantisation and asymmetric K/V quantisation without a format; this is
    the library's own): value = code * 2^(e - 127) with one exponent byte e
    per token and head (e = 0: zero).  codes: uint8 [..][64][D] (int8, two's
    complement) or [..][64][D/2] (int4 pairs, low nibble = even dim);
    v_exp: uint8 [..][64].  Returns the values as 16-bit storage bits of dtype;
    every value is exact there (7 significant bits at most), which is checked."""
    codes = np.asarray(codes, np.uint8)
    if v_format == V_INT8:
        q = codes.view(np.int8).astype(np.float64)
    elif v_format == V_INT4:
        lo = (codes & 0x0F).astype(np.int64)
        hi = (codes >> 4).astype(np.int64)
        lo = np.where(lo >= 8, lo - 16, lo)
        hi = np.where(hi >= 8, hi - 16, hi)
        q = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (2 * codes.shape[-1],)).astype(np.float64)
    else:
        raise ValueError(v_format)
    e = np.asarray(v_exp, np.int64)
    scale = np.where(e == 0, 0.0, np.ldexp(1.0, e - 127))
    val = q * scale[..., None]
    if dtype == BF16:
        bits32 = val.astype(np.float32).view(np.uint32)
        if np.any(bits32 & 0xFFFF) or not np.array_equal(bits32.view(np.float32).astype(np.float64), val):
            raise ValueError("value not exact in bf16")
        return (bits32 >> 16).astype(np.uint16)
    h = val.astype(np.float16)
    if not np.array_equal(h.astype(np.float64), val):
        raise ValueError("value not exact in fp16")
    return h.view(np.uint16)


def decode_e4m3(codes) -> np.ndarray:
    """FP8 E4M3 (the OCP 8-bit floating-point format: 1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN) to
    float64, from the format's definition: exponent field 0 gives subnormals
    (m / 8) * 2^-6, otherwise (1 + m / 8) * 2^(E - 7)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 0xF) & (m == 7), np.nan, mag)
    return sign * mag


def dequant_k_e4m3(codes, k_exp, dtype: int) -> np.ndarray:
    """Quantised K storage (a reading for the asymmetric K/V quantisation the
    pages list; the library's own format): value = e4m3(code) * 2^(e - 127)
    with one exponent byte e per token and head (e = 0: zero).  codes: uint8
    [..][64][D]; k_exp: uint8 [..][64].  Returns 16-bit storage bits of dtype;
    exact (4 significant bits) where the value is in the dtype's range, which
    is checked."""
    val = decode_e4m3(codes)
    e = np.asarray(k_exp, np.int64)
    scale = np.where(e == 0, 0.0, np.ldexp(1.0, e - 127))
    val = val * scale[..., None]
    if np.isnan(val).any():
        raise ValueError("NaN code in quantised K")
    if dtype == BF16:
        bits32 = val.astype(np.float32).view(np.uint32)
        if np.any(bits32 & 0xFFFF) or not np.array_equal(bits32.view(np.float32).astype(np.float64), val):
            raise ValueError("value not exact in bf16")
        return (bits32 >> 16).astype(np.uint16)
    h = val.astype(np.float16)
    if not np.array_equal(h.astype(np.float64), val):
        raise ValueError("value not exact in fp16")
    return h.view(np.uint16)


def _bits_to_f64(bits, dtype: int) -> np.ndarray:
    """16-bit storage bits of dtype to float64 (exact)."""
    b = np.asarray(bits, np.uint16)
    if dtype == BF16:
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return b.view(np.float16).astype(np.float64)


def _round_e4m3(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code to each |y| <= 448, ties to the even code (the codes of
    two neighbouring values differ by one, so exactly one is even); the sign
    bit follows y's sign bit."""
    pos = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: the non-negative finite codes, ascending
    vals = decode_e4m3(pos)
    a = np.abs(y)
    if np.any(a > 448.0):
        raise ValueError("beyond E4M3's range")
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = (d_lo == d_hi) & (lo != hi)
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    return (pos[pick] | np.where(np.signbit(y), 0x80, 0x00)).astype(np.uint8)


def quantise_k_e4m3(k_bits, dtype: int):
    """The storing side of the quantised-K format (the library's own reading of
    the asymmetric K/V quantisation the pages list without a format): for each
    token and head row k of 16-bit values, p is the largest integer with
    max|k| * 2^p <= 448 (E4M3's largest finite value), the exponent byte is
    e = 127 - p, and code d = e4m3(k_d * 2^p) rounded to nearest, ties to the
    even code.  An all-zero row gets e = 0 and zero codes.  k_bits: uint16
    [..][D]; returns (codes uint8 [..][D], k_exp uint8 [..]), which
    dequant_k_e4m3 reads back.  Raises if e would leave [1, 254]."""
    x = _bits_to_f64(k_bits, dtype)
    m = np.abs(x).max(axis=-1)
    mant, ex = np.frexp(m)                          # m = mant * 2^ex, mant in [0.5, 1)
    p = np.where(mant <= 0.875, 9 - ex, 8 - ex)     # 448 = 0.875 * 2^9
    zero = m == 0
    p = np.where(zero, 0, p).astype(np.int64)
    e = np.where(zero, 0, 127 - p)
    if np.any(~zero & ((e < 1) | (e > 254))):
        raise ValueError("row scale outside the exponent byte's range")
    codes = _round_e4m3(x * np.ldexp(1.0, p)[..., None])
    return codes, e.astype(np.uint8)


def commit_kq(inp: dict, k_codes, k_exp, acc_nodes, acc_len, inplace: bool = False):
    """Commit / rollback into a K pool held in the quantised-K format (V stays
    16-bit and goes through ``commit``): the k-th accepted node's K row of
    every KV head is stored at logical position L_b + k (pool page
    page_table[b][(L_b+k)/64], slot (L_b+k) % 64) as quantise_k_e4m3 of that
    16-bit row; every other code and exponent byte is unchanged.  k_codes
    uint8 [P][Hkv][64][D], k_exp uint8 [P][Hkv][64].  Returns (k_codes, k_exp),
    on copies unless ``inplace``."""
    dtype = inp.get("dtype_id", BF16)
    codes = k_codes if inplace else np.array(k_codes, dtype=np.uint8, copy=True)
    expo = k_exp if inplace else np.array(k_exp, dtype=np.uint8, copy=True)
    kt = np.asarray(inp["k_tree"], np.uint16)
    pt = np.asarray(inp["page_table"], np.int32)
    ctx = np.asarray(inp["ctx_len"], np.int32)
    acc = np.asarray(acc_nodes, np.int32)
    alen = np.asarray(acc_len, np.int32)
    B = kt.shape[0]
    for b in range(B):
        for k in range(int(alen[b])):
            node = int(acc[b, k])
            pos = int(ctx[b]) + k
            page = int(pt[b, pos // 64])
            c, e = quantise_k_e4m3(kt[b, node], dtype)   # one row per KV head
            codes[page, :, pos % 64, :] = c
            expo[page, :, pos % 64] = e
    return codes, expo
