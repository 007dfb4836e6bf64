"""CPU oracle for relay decode attention -- TEST INFRASTRUCTURE ONLY.

Plain fp64 C (oracle.c) behind ctypes.  Only tests/, __graft_entry__.smoke()
and bench.py's CPU-baseline / reference legs may import this package; the
library under shared_prompt_decode_gb300/ never does.

Functions:
    build()                         compile oracle.c -> oracle/_build/liboracle.so
    attention_rows(case, rows, part) fp64 attention for selected (b, i, h) rows
    attention_full(case, part)       every valid row, as [B, Lq, H, D] / [B, Lq, H]
    relay_fuse(...)                  the relay-fusion step on fp64 partials
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

PART = {"full": 0, "sys": 1, "ctx": 2}


class _Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Lq", ctypes.c_int32), ("H", ctypes.c_int32),
                ("D", ctypes.c_int32), ("Ls", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("scale", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # RELAY_ORACLE_LIB: a copy of the oracle with a mistake planted in
            # it, built by tests/test_oracle_mutations.py to show that the pins
            # catch it; unset, the oracle is built from oracle.c as it stands
            path = os.environ.get("RELAY_ORACLE_LIB")
            if not path:
                build()
                path = _LIB_PATH
            lib = ctypes.CDLL(path)
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_kv_append.restype = ctypes.c_int
            lib.oracle_sys_prefill.restype = ctypes.c_int
            lib.oracle_rope.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def _u16(t):
    """fp16 torch tensor / numpy array -> contiguous uint16 bit patterns."""
    if hasattr(t, "numpy"):
        t = t.contiguous().view(__import__("torch").int16).numpy()
    return np.ascontiguousarray(np.asarray(t).view(np.uint16))


def _i32(t):
    if t is None:
        return None
    if hasattr(t, "numpy"):
        t = t.numpy()
    return np.ascontiguousarray(np.asarray(t, dtype=np.int32))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def attention_rows(case, rows, part: str = "full", scale: float | None = None,
                   threads: int = 0, k_cache=None, v_cache=None, block_tables=None):
    """fp64 attention for the (b, i, h) rows given; returns (out [n, D], lse [n]).

    `case` is a synth.Case.  k_cache / v_cache / block_tables override the
    case's pool (e.g. a relabelled pool).
    """
    lib = _load()
    rows = list(rows)
    n = len(rows)
    D = case.D
    kc_ = k_cache if k_cache is not None else case.k_cache
    dims = _Dims(case.B, case.Lq, case.H, D, case.Ls, 16, kc_.shape[0],
                 (block_tables if block_tables is not None else case.block_tables).shape[1],
                 kc_.shape[1], float(1.0 / math.sqrt(D)) if scale is None else float(scale))
    rb = np.ascontiguousarray(np.array([r[0] for r in rows], dtype=np.int32))
    ri = np.ascontiguousarray(np.array([r[1] for r in rows], dtype=np.int32))
    rh = np.ascontiguousarray(np.array([r[2] for r in rows], dtype=np.int32))
    out = np.zeros((max(n, 1), D), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    q = _u16(case.q)
    sk = _u16(case.sys_k) if case.Ls > 0 else np.zeros(1, np.uint16)
    sv = _u16(case.sys_v) if case.Ls > 0 else np.zeros(1, np.uint16)
    kc = _u16(k_cache if k_cache is not None else case.k_cache)
    vc = _u16(v_cache if v_cache is not None else case.v_cache)
    bt = _i32(block_tables if block_tables is not None else case.block_tables)
    cl = _i32(case.ctx_lens)
    ql = _i32(case.q_lens)
    rc = lib.oracle_attention_rows(ctypes.byref(dims), ctypes.c_int(PART[part]),
                                   _ptr(q), _ptr(sk), _ptr(sv), _ptr(kc), _ptr(vc),
                                   _ptr(bt), _ptr(cl), _ptr(ql), ctypes.c_int64(n),
                                   _ptr(rb), _ptr(ri), _ptr(rh), _ptr(out), _ptr(lse),
                                   ctypes.c_int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attention_rows failed with code {rc}")
    return out[:n], lse[:n]


def sys_prefill(q_sys, sys_k, sys_v, rows=None, scale=None, threads: int = 0):
    """Causal self-attention of the system prompt: q_sys [Ls, H, D], sys_k /
    sys_v [Ls, Hkv, D] (fp16 torch tensors).  rows: (t, h) pairs (default:
    all).  Returns (out [n, D], lse [n]) in fp64."""
    lib = _load()
    Ls, H, D = q_sys.shape
    Hkv = sys_k.shape[1]
    if rows is None:
        rows = [(t, h) for t in range(Ls) for h in range(H)]
    rows = list(rows)
    n = len(rows)
    dims = _Dims(1, Ls, H, D, Ls, 16, 0, 0, Hkv, float(1.0 / math.sqrt(D)) if scale is None else float(scale))
    rt = np.ascontiguousarray(np.array([r[0] for r in rows], dtype=np.int32))
    rh = np.ascontiguousarray(np.array([r[1] for r in rows], dtype=np.int32))
    out = np.zeros((max(n, 1), D), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    rc = lib.oracle_sys_prefill(ctypes.byref(dims), _ptr(_u16(q_sys)), _ptr(_u16(sys_k)), _ptr(_u16(sys_v)),
                                ctypes.c_int64(n), _ptr(rt), _ptr(rh), _ptr(out), _ptr(lse), ctypes.c_int(threads))
    if rc != 0:
        raise ValueError(f"oracle_sys_prefill failed with code {rc}")
    return out[:n], lse[:n]


def rope(x, Ls, ctx_lens, q_lens=None, base=10000.0):
    """x [B, Lq, heads, D] fp16 rotated at positions Ls + ctx_lens[b] - q_lens[b] + i
    (rotate-half pairs j, j + D/2; angle p * base^(-2j/D)); fp64 result, padding rows NaN."""
    lib = _load()
    B, Lq, heads, D = x.shape
    out = np.zeros((B, Lq, heads, D), dtype=np.float64)
    dims = _Dims(B, Lq, heads, D, int(Ls), 16, 0, 0, 1, 0.0)
    rc = lib.oracle_rope(ctypes.byref(dims), ctypes.c_double(base), ctypes.c_int(heads), _ptr(_i32(ctx_lens)),
                         _ptr(_i32(q_lens)), _ptr(_u16(x)), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_rope failed with code {rc}")
    return out


def kv_append(case, k_new, v_new):
    """The case's pools after appending k_new / v_new ([B, Lq, Hkv, D] fp16)
    at each request's last q_lens[b] context positions; returns new torch
    tensors (the case is not modified)."""
    import torch
    lib = _load()
    kc = _u16(case.k_cache).copy()
    vc = _u16(case.v_cache).copy()
    dims = _Dims(case.B, case.Lq, case.H, case.D, case.Ls, 16, case.k_cache.shape[0], case.block_tables.shape[1],
                 case.k_cache.shape[1], 0.0)
    rc = lib.oracle_kv_append(ctypes.byref(dims), _ptr(_u16(k_new)), _ptr(_u16(v_new)), _ptr(_i32(case.block_tables)),
                              _ptr(_i32(case.ctx_lens)), _ptr(_i32(case.q_lens)), _ptr(kc), _ptr(vc))
    if rc != 0:
        raise ValueError(f"oracle_kv_append failed with code {rc}")
    to_t = lambda a: torch.from_numpy(a.view(np.int16).reshape(case.k_cache.shape)).view(torch.float16)
    return to_t(kc), to_t(vc)


def all_rows(case):
    ql = case.q_lens_list()
    return [(b, i, h) for b in range(case.B) for i in range(ql[b]) for h in range(case.H)]


def attention_full(case, part: str = "full", scale: float | None = None, threads: int = 0):
    """Every valid row: out [B, Lq, H, D] and lse [B, Lq, H]; padding rows are NaN."""
    rows = all_rows(case)
    o, l = attention_rows(case, rows, part, scale, threads)
    out = np.full((case.B, case.Lq, case.H, case.D), np.nan)
    lse = np.full((case.B, case.Lq, case.H), np.nan)
    if rows:
        idx = np.array(rows)
        out[idx[:, 0], idx[:, 1], idx[:, 2]] = o
        lse[idx[:, 0], idx[:, 1], idx[:, 2]] = l
    return out, lse


def relay_fuse(o_sys, lse_sys, o_ctx, lse_ctx):
    """Relay fusion of fp64 partials; returns (out, lse, alpha_sys)."""
    lib = _load()
    o_sys = np.ascontiguousarray(o_sys, dtype=np.float64)
    o_ctx = np.ascontiguousarray(o_ctx, dtype=np.float64)
    lse_sys = np.ascontiguousarray(lse_sys, dtype=np.float64)
    lse_ctx = np.ascontiguousarray(lse_ctx, dtype=np.float64)
    shape = lse_sys.shape
    D = o_sys.shape[-1]
    n = int(np.prod(shape)) if shape else 1
    out = np.zeros_like(o_sys)
    lse = np.zeros_like(lse_sys)
    alpha = np.zeros_like(lse_sys)
    lib.oracle_relay_fuse(ctypes.c_int64(n), ctypes.c_int(D), _ptr(o_sys), _ptr(lse_sys),
                          _ptr(o_ctx), _ptr(lse_ctx), _ptr(out), _ptr(lse), _ptr(alpha))
    return out, lse, alpha


def half_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.zeros(bits.shape, dtype=np.float64)
    lib.oracle_half_to_double(ctypes.c_int64(bits.size), _ptr(bits), _ptr(out))
    return out
