"""Relay decode attention on GB300: thin Python binding of librelay.so.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of librelay.so (built from csrc/ by build.py).  torch supplies device
memory and the current stream.  There is no CPU or PyTorch fallback: if the
library is missing, importing the binding's functions raises.

Entry points (same names as the C ABI in include/relay.h):
    relay_attention_decode(...)   all three steps, queued as one unit (two kernels; three with
                                  the tensor-core system step)
    relay_attention_decode_prefixes(...)  the same for a tree of shared prefixes: several shared
                                  segments, each request seeing those its mask selects
    relay_sys_attn(...)           step 1: system attention -> fp32 o, lse
    relay_ctx_attn(...)           step 2: context attention -> fp32 o, lse
    relay_fuse(...)               step 3: relay fusion -> fp16 out, lse
    relay_fuse_n(...)             relay fusion of K parts (a tree of shared prefixes)
    relay_baseline_decode(...)    non-relay paged attention over [system; context]
    relay_kv_append(...)          the step's new K/V rows into the paged pool
    relay_sys_prefill(...)        causal self-attention of the system prompt (filling its cache)
    relay_rope(...)               rotary positions of the new rows, offset by the system prompt
    workspace_size(dims), make_workspace(dims), device_status(ws)
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librelay.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT = range(7)
FLAG_BAD_Q_LEN, FLAG_BAD_CTX_LEN, FLAG_BAD_BLOCK, FLAG_Q_TOTAL, FLAG_WAIT_TIMEOUT = 1, 2, 4, 8, 16


class RelayError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("Lq", ctypes.c_int32), ("H", ctypes.c_int32),
                ("D", ctypes.c_int32), ("Ls", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("max_q_total", ctypes.c_int32), ("ctx_split", ctypes.c_int32),
                ("sys_range", ctypes.c_int32), ("scale", ctypes.c_float), ("Hkv", ctypes.c_int32)]

    def __repr__(self):
        return "Dims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_lib = None

_VP = ctypes.c_void_p
_SIGS = {
    "relay_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Dims)]),
    "relay_workspace_init": (ctypes.c_int, [_VP, ctypes.c_size_t, _VP]),
    "relay_sys_attn": (ctypes.c_int, [ctypes.POINTER(Dims), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                      ctypes.c_size_t, _VP]),
    "relay_ctx_attn": (ctypes.c_int, [ctypes.POINTER(Dims), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                      _VP, ctypes.c_size_t, _VP]),
    "relay_fuse": (ctypes.c_int, [ctypes.POINTER(Dims), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "relay_attention_decode": (ctypes.c_int, [ctypes.POINTER(Dims)] + [_VP] * 11 + [ctypes.c_size_t, _VP]),
    "relay_baseline_decode": (ctypes.c_int, [ctypes.POINTER(Dims)] + [_VP] * 10 + [ctypes.c_size_t, _VP]),
    "relay_device_status": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_uint32), _VP]),
    "relay_kv_append": (ctypes.c_int, [ctypes.POINTER(Dims)] + [_VP] * 8 + [ctypes.c_size_t, _VP]),
    "relay_sys_prefill": (ctypes.c_int, [ctypes.POINTER(Dims)] + [_VP] * 6 + [ctypes.c_size_t, _VP]),
    "relay_fuse_n": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_int, _VP, _VP, _VP, _VP, _VP, _VP]),
    "relay_rope": (ctypes.c_int, [ctypes.POINTER(Dims)] + [_VP] * 4 + [ctypes.c_float, _VP, ctypes.c_size_t, _VP]),
    "relay_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "relay_workspace_size_prefixes": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int, _VP]),
    "relay_attention_decode_prefixes": (ctypes.c_int, [ctypes.POINTER(Dims), _VP, ctypes.c_int, _VP, _VP, _VP, _VP]
                                        + [_VP] * 8 + [ctypes.c_size_t, _VP]),
}


def lib():
    """The loaded librelay.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librelay.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().relay_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != OK:
        raise RelayError(code, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _shape(t, name, shape):
    """Shape check of a tensor the kernels index by the dims (an optional one may be None); done before the
    device checks, so that a wrong size never reaches the library as a plain pointer."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _same(a, b, names):
    if tuple(a.shape) != tuple(b.shape):
        raise ValueError(f"{names[0]} {tuple(a.shape)} and {names[1]} {tuple(b.shape)} must have the same shape")


def _opt(t, name, dtype, device):
    if t is not None:
        _need(t, name, dtype, device)


def _check_dims(dims: Dims, q, Ls=None, pool=None, block_tables=None):
    """Explicit dims must describe the tensors: the kernels take every size and stride from them."""
    B, Lq, H, D = q.shape
    if (dims.B, dims.Lq, dims.H, dims.D) != (B, Lq, H, D):
        raise ValueError(f"dims {dims} do not match q {tuple(q.shape)}")
    if Ls is not None and dims.Ls != Ls:
        raise ValueError(f"dims.Ls = {dims.Ls}, but the system cache holds {Ls} tokens")
    if pool is not None and dims.num_blocks > pool.shape[0]:
        raise ValueError(f"dims.num_blocks = {dims.num_blocks} exceeds the pool's {pool.shape[0]} blocks")
    if block_tables is not None and dims.max_blocks_per_seq != block_tables.shape[1]:
        raise ValueError(f"dims.max_blocks_per_seq = {dims.max_blocks_per_seq}, but block_tables rows hold "
                         f"{block_tables.shape[1]} entries")


def _pool_shapes(k, v, D, names):
    _same(k, v, names)
    if k.dim() != 4 or k.shape[2] != 16 or k.shape[3] != D:
        raise ValueError(f"{names[0]} {tuple(k.shape)} must be [num_blocks, Hkv, 16, {D}]")


def _table_shapes(B, block_tables, ctx_lens, q_lens):
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError(f"block_tables {tuple(block_tables.shape)} must be [{B}, max_blocks]")
    _shape(ctx_lens, "ctx_lens", (B,))
    _shape(q_lens, "q_lens", (B,))


def make_dims(q: torch.Tensor, Ls: int, num_blocks: int, max_blocks: int, scale: Optional[float] = None,
              max_q_total: int = 0, ctx_split: int = 0, sys_range: int = 0, Hkv: int = 0) -> Dims:
    """Hkv: KV heads of the caches (0: as many as query heads)."""
    B, Lq, H, D = q.shape
    return Dims(B, Lq, H, D, Ls, 16, num_blocks, max_blocks, max_q_total, ctx_split, sys_range,
                0.0 if scale is None else float(scale), Hkv)


def _check_kv(dims: Dims, cache: torch.Tensor, name: str):
    """The cache's head dimension (dim 1) must be the dims' KV heads."""
    hkv = dims.Hkv if dims.Hkv > 0 else dims.H
    if cache.dim() < 3 or cache.shape[1] != hkv:
        raise ValueError(f"{name} has {cache.shape[1] if cache.dim() > 1 else '?'} KV heads, dims say {hkv}")


def workspace_size(dims: Dims) -> int:
    return int(lib().relay_workspace_size(ctypes.byref(dims)))


def make_workspace(dims: Dims, device=None) -> torch.Tensor:
    """Zero-filled workspace of the size `dims` needs (torch owns the memory)."""
    n = workspace_size(dims)
    if n == 0:
        raise ValueError(f"invalid dims {dims}")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ws(dims, workspace, device):
    if workspace is None:
        workspace = make_workspace(dims, device)
    return workspace


def relay_attention_decode(q, sys_k, sys_v, k_cache, v_cache, block_tables, ctx_lens, q_lens=None,
                           out=None, lse_out=None, workspace=None, scale=None, max_q_total=0,
                           ctx_split=0, sys_range=0, stream=None, dims=None):
    """All three steps, queued as one unit on the stream.  Returns out [B, Lq, H, D] fp16."""
    dev = q.device
    B, Lq, H, D = q.shape
    _same(sys_k, sys_v, ("sys_k", "sys_v"))
    if sys_k.dim() != 3 or sys_k.shape[2] != D:
        raise ValueError(f"sys_k {tuple(sys_k.shape)} must be [Ls, Hkv, {D}]")
    _pool_shapes(k_cache, v_cache, D, ("k_cache", "v_cache"))
    _table_shapes(B, block_tables, ctx_lens, q_lens)
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", (B, Lq, H))
    _need(q, "q", torch.float16)
    for name, t in (("sys_k", sys_k), ("sys_v", sys_v), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, torch.float16, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    if dims is None:
        dims = make_dims(q, sys_k.shape[0], k_cache.shape[0], block_tables.shape[1], scale,
                         max_q_total, ctx_split, sys_range, k_cache.shape[1])
    _check_dims(dims, q, sys_k.shape[0], k_cache, block_tables)
    _check_kv(dims, sys_k, "sys_k")
    _check_kv(dims, k_cache, "k_cache")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, dev)
    _opt(lse_out, "lse_out", torch.float32, dev)
    ws = _ws(dims, workspace, dev)
    rc = lib().relay_attention_decode(ctypes.byref(dims), _ptr(q), _ptr(sys_k), _ptr(sys_v), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens),
                                      _ptr(out), _ptr(lse_out), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "relay_attention_decode")
    return out


MAX_SEGMENTS = 8


def prefixes_workspace_size(dims: Dims, seg_lens) -> int:
    arr = (ctypes.c_int32 * len(seg_lens))(*[int(x) for x in seg_lens])
    return int(lib().relay_workspace_size_prefixes(ctypes.byref(dims), len(seg_lens), arr))


def relay_attention_decode_prefixes(q, seg_k, seg_v, seg_mask, k_cache, v_cache, block_tables, ctx_lens,
                                    q_lens=None, out=None, lse_out=None, workspace=None, scale=None,
                                    max_q_total=0, ctx_split=0, sys_range=0, stream=None, dims=None):
    """A tree of shared prefixes: seg_k / seg_v are lists of [L_s, Hkv, D] fp16 segments, seg_mask a
    [B] int32 tensor whose bit s says that request b sees segment s (None: every request sees every
    segment).  Returns out [B, Lq, H, D] fp16."""
    dev = q.device
    B, Lq, H, D = q.shape
    if not (1 <= len(seg_k) <= MAX_SEGMENTS) or len(seg_k) != len(seg_v):
        raise ValueError(f"1..{MAX_SEGMENTS} segments with K and V each")
    Hkv = k_cache.shape[1]
    for i, (k, v) in enumerate(zip(seg_k, seg_v)):
        _same(k, v, (f"seg_k[{i}]", f"seg_v[{i}]"))
        if k.dim() != 3 or k.shape[1] != Hkv or k.shape[2] != D:
            raise ValueError(f"seg_k[{i}] {tuple(k.shape)} must be [L, {Hkv}, {D}]")
        _need(k, f"seg_k[{i}]", torch.float16, dev)
        _need(v, f"seg_v[{i}]", torch.float16, dev)
    _pool_shapes(k_cache, v_cache, D, ("k_cache", "v_cache"))
    _table_shapes(B, block_tables, ctx_lens, q_lens)
    _shape(seg_mask, "seg_mask", (B,))
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", (B, Lq, H))
    _need(q, "q", torch.float16)
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, torch.float16, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(seg_mask, "seg_mask", torch.int32, dev)
    if dims is None:
        dims = make_dims(q, 0, k_cache.shape[0], block_tables.shape[1], scale, max_q_total, ctx_split, sys_range,
                         Hkv)
    _check_dims(dims, q, None, k_cache, block_tables)
    _check_kv(dims, k_cache, "k_cache")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.float16, dev)
    _opt(lse_out, "lse_out", torch.float32, dev)
    lens = [int(k.shape[0]) for k in seg_k]
    if workspace is None:
        n = prefixes_workspace_size(dims, lens)
        if n == 0:
            raise ValueError(f"invalid dims {dims} or segments {lens}")
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    n = len(seg_k)
    kp = (ctypes.c_void_p * n)(*[k.data_ptr() for k in seg_k])
    vp = (ctypes.c_void_p * n)(*[v.data_ptr() for v in seg_v])
    lp = (ctypes.c_int32 * n)(*lens)
    rc = lib().relay_attention_decode_prefixes(
        ctypes.byref(dims), _ptr(q), n, kp, vp, lp, _ptr(seg_mask), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens), _ptr(out), _ptr(lse_out), _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check(rc, "relay_attention_decode_prefixes")
    return out


def relay_sys_attn(q, sys_k, sys_v, q_lens=None, o_sys=None, lse_sys=None, workspace=None, scale=None,
                   max_q_total=0, sys_range=0, stream=None, max_blocks=0):
    dev = q.device
    B, Lq, H, D = q.shape
    _same(sys_k, sys_v, ("sys_k", "sys_v"))
    if sys_k.dim() != 3 or sys_k.shape[2] != D:
        raise ValueError(f"sys_k {tuple(sys_k.shape)} must be [Ls, Hkv, {D}]")
    _shape(q_lens, "q_lens", (B,))
    _shape(o_sys, "o_sys", q.shape)
    _shape(lse_sys, "lse_sys", (B, Lq, H))
    _need(q, "q", torch.float16)
    _need(sys_k, "sys_k", torch.float16, dev)
    _need(sys_v, "sys_v", torch.float16, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(o_sys, "o_sys", torch.float32, dev)
    _opt(lse_sys, "lse_sys", torch.float32, dev)
    dims = make_dims(q, sys_k.shape[0], 0, max_blocks, scale, max_q_total, 0, sys_range, sys_k.shape[1])
    if o_sys is None:
        o_sys = torch.empty(B, Lq, H, D, dtype=torch.float32, device=dev)
    if lse_sys is None:
        lse_sys = torch.empty(B, Lq, H, dtype=torch.float32, device=dev)
    ws = _ws(dims, workspace, dev)
    rc = lib().relay_sys_attn(ctypes.byref(dims), _ptr(q), _ptr(sys_k), _ptr(sys_v), _ptr(q_lens), _ptr(o_sys),
                              _ptr(lse_sys), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "relay_sys_attn")
    return o_sys, lse_sys


def relay_ctx_attn(q, k_cache, v_cache, block_tables, ctx_lens, q_lens=None, o_ctx=None, lse_ctx=None,
                   workspace=None, scale=None, max_q_total=0, ctx_split=0, stream=None):
    dev = q.device
    B, Lq, H, D = q.shape
    _pool_shapes(k_cache, v_cache, D, ("k_cache", "v_cache"))
    _table_shapes(B, block_tables, ctx_lens, q_lens)
    _shape(o_ctx, "o_ctx", q.shape)
    _shape(lse_ctx, "lse_ctx", (B, Lq, H))
    _need(q, "q", torch.float16)
    _need(k_cache, "k_cache", torch.float16, dev)
    _need(v_cache, "v_cache", torch.float16, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(o_ctx, "o_ctx", torch.float32, dev)
    _opt(lse_ctx, "lse_ctx", torch.float32, dev)
    dims = make_dims(q, 0, k_cache.shape[0], block_tables.shape[1], scale, max_q_total, ctx_split, 0,
                     k_cache.shape[1])
    if o_ctx is None:
        o_ctx = torch.empty(B, Lq, H, D, dtype=torch.float32, device=dev)
    if lse_ctx is None:
        lse_ctx = torch.empty(B, Lq, H, dtype=torch.float32, device=dev)
    ws = _ws(dims, workspace, dev)
    rc = lib().relay_ctx_attn(ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              _ptr(ctx_lens), _ptr(q_lens), _ptr(o_ctx), _ptr(lse_ctx), _ptr(ws), ws.numel(),
                              _stream(stream))
    _check(rc, "relay_ctx_attn")
    return o_ctx, lse_ctx


def relay_fuse(o_sys, lse_sys, o_ctx, lse_ctx, q_lens=None, out=None, lse_out=None, stream=None):
    dev = o_sys.device
    B, Lq, H, D = o_sys.shape
    _shape(o_ctx, "o_ctx", o_sys.shape)
    _shape(lse_sys, "lse_sys", (B, Lq, H))
    _shape(lse_ctx, "lse_ctx", (B, Lq, H))
    _shape(q_lens, "q_lens", (B,))
    _shape(out, "out", o_sys.shape)
    _shape(lse_out, "lse_out", (B, Lq, H))
    for name, t in (("o_sys", o_sys), ("lse_sys", lse_sys), ("o_ctx", o_ctx), ("lse_ctx", lse_ctx)):
        _need(t, name, torch.float32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(out, "out", torch.float16, dev)
    _opt(lse_out, "lse_out", torch.float32, dev)
    dims = Dims(B, Lq, H, D, 0, 16, 0, 0, 0, 0, 0, 0.0)
    if out is None:
        out = torch.empty(B, Lq, H, D, dtype=torch.float16, device=dev)
    rc = lib().relay_fuse(ctypes.byref(dims), _ptr(o_sys), _ptr(lse_sys), _ptr(o_ctx), _ptr(lse_ctx), _ptr(q_lens),
                          _ptr(out), _ptr(lse_out), _stream(stream))
    _check(rc, "relay_fuse")
    return out


def relay_fuse_n(o_parts, lse_parts, q_lens=None, out=None, lse_out=None, stream=None):
    """Relay fusion of K partial results (lists of [B, Lq, H, D] / [B, Lq, H] fp32 tensors)."""
    K = len(o_parts)
    if K != len(lse_parts) or K < 1:
        raise ValueError("o_parts and lse_parts must be non-empty and of the same length")
    dev = o_parts[0].device
    B, Lq, H, D = o_parts[0].shape
    for k in range(K):
        _shape(o_parts[k], f"o_parts[{k}]", (B, Lq, H, D))
        _shape(lse_parts[k], f"lse_parts[{k}]", (B, Lq, H))
    _shape(q_lens, "q_lens", (B,))
    _shape(out, "out", (B, Lq, H, D))
    _shape(lse_out, "lse_out", (B, Lq, H))
    for k in range(K):
        _need(o_parts[k], f"o_parts[{k}]", torch.float32, dev)
        _need(lse_parts[k], f"lse_parts[{k}]", torch.float32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(out, "out", torch.float16, dev)
    _opt(lse_out, "lse_out", torch.float32, dev)
    dims = Dims(B, Lq, H, D, 0, 16, 0, 0, 0, 0, 0, 0.0)
    if out is None:
        out = torch.empty(B, Lq, H, D, dtype=torch.float16, device=dev)
    op = (ctypes.c_void_p * K)(*[t.data_ptr() for t in o_parts])
    lp = (ctypes.c_void_p * K)(*[t.data_ptr() for t in lse_parts])
    rc = lib().relay_fuse_n(ctypes.byref(dims), K, ctypes.cast(op, ctypes.c_void_p), ctypes.cast(lp, ctypes.c_void_p),
                            _ptr(q_lens), _ptr(out), _ptr(lse_out), _stream(stream))
    _check(rc, "relay_fuse_n")
    return out


def relay_baseline_decode(q, k_pool, v_pool, sys_block_ids, Ls, block_tables, ctx_lens, q_lens=None,
                          out=None, lse_out=None, workspace=None, scale=None, max_q_total=0, ctx_split=0,
                          stream=None, dims=None):
    dev = q.device
    B, Lq, H, D = q.shape
    _pool_shapes(k_pool, v_pool, D, ("k_pool", "v_pool"))
    _table_shapes(B, block_tables, ctx_lens, q_lens)
    if sys_block_ids.dim() != 1 or sys_block_ids.shape[0] < (int(Ls) + 15) // 16:
        raise ValueError(f"sys_block_ids {tuple(sys_block_ids.shape)} must list the {(int(Ls) + 15) // 16} "
                         f"blocks of the {int(Ls)} system tokens")
    _shape(out, "out", q.shape)
    _shape(lse_out, "lse_out", (B, Lq, H))
    _need(q, "q", torch.float16)
    _need(k_pool, "k_pool", torch.float16, dev)
    _need(v_pool, "v_pool", torch.float16, dev)
    _need(sys_block_ids, "sys_block_ids", torch.int32, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    _opt(out, "out", torch.float16, dev)
    _opt(lse_out, "lse_out", torch.float32, dev)
    if dims is None:
        dims = make_dims(q, Ls, k_pool.shape[0], block_tables.shape[1], scale, max_q_total, ctx_split, 0,
                         k_pool.shape[1])
    _check_dims(dims, q, int(Ls), k_pool, block_tables)
    _check_kv(dims, k_pool, "k_pool")
    if out is None:
        out = torch.empty_like(q)
    ws = _ws(dims, workspace, dev)
    rc = lib().relay_baseline_decode(ctypes.byref(dims), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(sys_block_ids),
                                     _ptr(block_tables), _ptr(ctx_lens), _ptr(q_lens), _ptr(out), _ptr(lse_out),
                                     _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "relay_baseline_decode")
    return out


def relay_kv_append(k_new, v_new, block_tables, ctx_lens, k_cache, v_cache, q_lens=None, workspace=None,
                    stream=None):
    """Write the step's new K/V rows ([B, Lq, Hkv, D] fp16) into the paged pools in place, at each request's
    last q_lens[b] context positions.  Device-side problems are flagged in `workspace` (device_status)."""
    dev = k_new.device
    B, Lq, Hkv, D = k_new.shape
    if v_new.shape != k_new.shape or k_cache.shape != v_cache.shape or k_cache.dim() != 4 or \
            k_cache.shape[1] != Hkv or k_cache.shape[2] != 16 or k_cache.shape[3] != D:
        raise ValueError("k_new/v_new [B, Lq, Hkv, D] and the pools [num_blocks, Hkv, 16, D] disagree")
    _table_shapes(B, block_tables, ctx_lens, q_lens)
    _need(k_new, "k_new", torch.float16)
    for name, t in (("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, torch.float16, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    dims = Dims(B, Lq, Hkv, D, 0, 16, k_cache.shape[0], block_tables.shape[1], 0, 0, 0, 0.0, Hkv)
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=dev)
    rc = lib().relay_kv_append(ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(block_tables), _ptr(ctx_lens),
                               _ptr(q_lens), _ptr(k_cache), _ptr(v_cache), _ptr(workspace), workspace.numel(),
                               _stream(stream))
    _check(rc, "relay_kv_append")
    return workspace


def relay_sys_prefill(q_sys, sys_k, sys_v, out=None, lse_out=None, workspace=None, scale=None, stream=None):
    """Causal self-attention of the system prompt (the attention step of filling its cache offline):
    q_sys [Ls, H, 128] fp16, sys_k / sys_v [Ls, Hkv, 128] fp16 -> out [Ls, H, 128] fp16 (and lse_out [Ls, H])."""
    dev = q_sys.device
    Ls, H, D = q_sys.shape
    if sys_k.shape != sys_v.shape or sys_k.dim() != 3 or sys_k.shape[0] != Ls or sys_k.shape[2] != D:
        raise ValueError("q_sys [Ls, H, D] and sys_k / sys_v [Ls, Hkv, D] disagree")
    _shape(out, "out", q_sys.shape)
    _shape(lse_out, "lse_out", (Ls, H))
    _need(q_sys, "q_sys", torch.float16)
    _need(sys_k, "sys_k", torch.float16, dev)
    _need(sys_v, "sys_v", torch.float16, dev)
    dims = Dims(1, 1, H, D, Ls, 16, 0, 0, 0, 0, 0, 0.0 if scale is None else float(scale), sys_k.shape[1])
    if out is None:
        out = torch.empty_like(q_sys)
    _need(out, "out", torch.float16, dev)
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, dev)
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=dev)
    rc = lib().relay_sys_prefill(ctypes.byref(dims), _ptr(q_sys), _ptr(sys_k), _ptr(sys_v), _ptr(out), _ptr(lse_out),
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "relay_sys_prefill")
    return out


def relay_rope(q, ctx_lens, Ls, k_new=None, q_lens=None, base=10000.0, workspace=None, stream=None):
    """Rotary embedding in place of q [B, Lq, H, D] (and k_new [B, Lq, Hkv, D]) at positions
    Ls + ctx_lens[b] - q_lens[b] + i: the request tokens follow the Ls system tokens."""
    dev = q.device
    B, Lq, H, D = q.shape
    Hkv = k_new.shape[2] if k_new is not None else H
    if k_new is not None and (k_new.dim() != 4 or tuple(k_new.shape) != (B, Lq, Hkv, D)):
        raise ValueError(f"k_new {tuple(k_new.shape)} must be [{B}, {Lq}, Hkv, {D}]")
    _shape(ctx_lens, "ctx_lens", (B,))
    _shape(q_lens, "q_lens", (B,))
    _need(q, "q", torch.float16)
    _need(ctx_lens, "ctx_lens", torch.int32, dev)
    _opt(k_new, "k_new", torch.float16, dev)
    _opt(q_lens, "q_lens", torch.int32, dev)
    dims = Dims(B, Lq, H, D, int(Ls), 16, 0, 0, 0, 0, 0, 0.0, Hkv)
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=dev)
    rc = lib().relay_rope(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(ctx_lens), _ptr(q_lens), float(base),
                          _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "relay_rope")
    return workspace


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Read and clear the device-side check flags (synchronises the stream)."""
    flags = ctypes.c_uint32(0)
    rc = lib().relay_device_status(_ptr(workspace), ctypes.byref(flags), _stream(stream))
    if rc not in (OK, ERR_DEVICE_CHECK):
        raise RelayError(rc, "relay_device_status")
    return int(flags.value)


def algorithmic_bytes(B, H, D, Ls, ctx_lens, q_rows, Hkv=None) -> int:
    """Bytes the relay step must move at minimum: the system KV once, every
    request's context KV once (Hkv heads), q read and out written (fp16)."""
    kv_token = 2 * (H if not Hkv else Hkv) * D * 2
    return Ls * kv_token + int(sum(int(n) for n in ctx_lens)) * kv_token + 2 * q_rows * H * D * 2
