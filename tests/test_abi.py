"""The C ABI without a GPU: the library loads, exports every declared symbol,
its struct layout matches the binding, and host-side validation rejects bad
arguments before anything is queued (no CUDA call is reached)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "relay.h")


@pytest.fixture(scope="module")
def relay():
    from shared_prompt_decode_gb300 import build
    build.build()
    import shared_prompt_decode_gb300 as r
    r.lib()
    return r


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(relay_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(relay):
    names = _declared()
    assert {"relay_attention_decode", "relay_sys_attn", "relay_ctx_attn", "relay_fuse",
            "relay_baseline_decode", "relay_workspace_size", "relay_status_string"} <= set(names)
    lib = ctypes.CDLL(relay.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_dims_layout_matches_header(relay, tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "relay.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(relay_dims_t),"
        " offsetof(relay_dims_t, max_q_total), offsetof(relay_dims_t, sys_range),"
        " offsetof(relay_dims_t, scale), offsetof(relay_dims_t, Hkv));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    D = relay.Dims
    assert got == [ctypes.sizeof(D), D.max_q_total.offset, D.sys_range.offset, D.scale.offset, D.Hkv.offset]


def test_status_strings(relay):
    for code in range(7):
        assert relay.status_string(code) and relay.status_string(code) != "unknown status"
    assert relay.status_string(99) == "unknown status"


def _dims(relay, **kw):
    base = dict(B=32, Lq=1, H=32, D=128, Ls=2048, block_size=16, num_blocks=1200, max_blocks_per_seq=64,
                max_q_total=0, ctx_split=0, sys_range=0, scale=0.0, Hkv=0)
    base.update(kw)
    return relay.Dims(**base)


def test_workspace_size(relay):
    lib = relay.lib()
    n = lib.relay_workspace_size(ctypes.byref(_dims(relay)))
    assert n > 0 and n % 256 == 0
    assert lib.relay_workspace_size(ctypes.byref(_dims(relay, B=64))) > n
    assert lib.relay_workspace_size(None) == 0
    for bad in (dict(D=96), dict(block_size=32), dict(B=513), dict(H=0), dict(Lq=0), dict(Ls=-1),
                dict(ctx_split=100), dict(sys_range=-64), dict(Hkv=-1), dict(Hkv=3), dict(Hkv=64)):
        assert lib.relay_workspace_size(ctypes.byref(_dims(relay, **bad))) == 0, bad
    # a bound on the total query rows shrinks the partial storage
    big = lib.relay_workspace_size(ctypes.byref(_dims(relay, B=64, Lq=128, H=40, Ls=32768, max_blocks_per_seq=256)))
    small = lib.relay_workspace_size(ctypes.byref(_dims(relay, B=64, Lq=128, H=40, Ls=32768, max_blocks_per_seq=256,
                                                        max_q_total=1080)))
    assert small < big / 4
    # grouped-query heads: any divisor of H is valid (the partials stay per
    # query head; the number of system key ranges follows the KV heads)
    for hkv in (1, 8, 32):
        m = lib.relay_workspace_size(ctypes.byref(_dims(relay, Hkv=hkv)))
        assert m > 0 and m % 256 == 0, hkv


FAKE = 0x7f0000000000      # never dereferenced: validation fails first


def _call_decode(relay, dims, ws_bytes=1 << 30, **over):
    args = dict(q=FAKE, sys_k=FAKE, sys_v=FAKE, k=FAKE, v=FAKE, bt=FAKE, cl=FAKE, ql=None, out=FAKE,
                lse=None, ws=FAKE)
    args.update(over)
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    return relay.lib().relay_attention_decode(
        ctypes.byref(dims) if dims is not None else None, vp(args["q"]), vp(args["sys_k"]), vp(args["sys_v"]),
        vp(args["k"]), vp(args["v"]), vp(args["bt"]), vp(args["cl"]), vp(args["ql"]), vp(args["out"]),
        vp(args["lse"]), vp(args["ws"]), ws_bytes, None)


def test_host_validation(relay):
    d = _dims(relay)
    assert _call_decode(relay, None) == relay.ERR_INVALID_ARG
    assert _call_decode(relay, _dims(relay, D=96)) == relay.ERR_UNSUPPORTED
    assert _call_decode(relay, _dims(relay, block_size=8)) == relay.ERR_UNSUPPORTED
    assert _call_decode(relay, _dims(relay, Hkv=5)) == relay.ERR_INVALID_ARG   # 32 query heads, 5 KV heads
    # grouped-query and multi-query heads pass the shape checks: the calls get as far as the pointer checks
    # (q missing) or, with nothing to do, return OK without queueing anything
    for hkv in (1, 2, 8, 16):
        assert _call_decode(relay, _dims(relay, Hkv=hkv), q=None) == relay.ERR_INVALID_ARG, hkv
        assert _call_decode(relay, _dims(relay, Hkv=hkv, B=0)) == relay.OK, hkv
    assert _call_decode(relay, _dims(relay, B=1024)) == relay.ERR_UNSUPPORTED
    assert _call_decode(relay, d, q=None) == relay.ERR_INVALID_ARG
    assert _call_decode(relay, d, out=None) == relay.ERR_INVALID_ARG
    assert _call_decode(relay, d, cl=None) == relay.ERR_INVALID_ARG
    assert _call_decode(relay, d, sys_k=None) == relay.ERR_INVALID_ARG
    assert _call_decode(relay, d, q=FAKE + 2) == relay.ERR_INVALID_ARG      # not 16-byte aligned
    assert _call_decode(relay, d, lse=FAKE + 2) == relay.ERR_INVALID_ARG    # not 4-byte aligned
    assert _call_decode(relay, d, ws=None) == relay.ERR_WORKSPACE
    assert _call_decode(relay, d, ws_bytes=1024) == relay.ERR_WORKSPACE
    assert _call_decode(relay, d, ws=FAKE + 16) == relay.ERR_INVALID_ARG    # workspace not 256-aligned
    # no q_lens: B * Lq rows, above a smaller max_q_total (with q_lens the device checks the sum)
    assert _call_decode(relay, _dims(relay, Lq=2, max_q_total=3)) == relay.ERR_INVALID_ARG
    # Ls == 0: the system cache may be absent; B == 0: nothing to do, nothing queued
    assert _call_decode(relay, _dims(relay, B=0)) == relay.OK
    lib = relay.lib()
    assert lib.relay_fuse(ctypes.byref(d), None, None, None, None, None, None, None, None) == relay.ERR_INVALID_ARG
    assert lib.relay_sys_attn(ctypes.byref(_dims(relay, D=80)), *([ctypes.c_void_p(FAKE)] * 7), 1 << 30,
                              None) == relay.ERR_UNSUPPORTED
    assert lib.relay_device_status(None, None, None) == relay.ERR_WORKSPACE


def test_kv_append_host_validation(relay):
    lib = relay.lib()
    d = _dims(relay, Lq=2)
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    call = lambda **o: lib.relay_kv_append(
        ctypes.byref(d), *[vp(o.get(k, FAKE)) for k in ("kn", "vn", "bt", "cl", "ql", "kc", "vc", "ws")],
        o.get("ws_bytes", 1 << 20), None)
    assert call(ws=None) == relay.ERR_WORKSPACE
    assert call(ws_bytes=128) == relay.ERR_WORKSPACE
    assert call(kn=None) == relay.ERR_INVALID_ARG
    assert call(kc=None) == relay.ERR_INVALID_ARG
    assert call(kn=FAKE + 8) == relay.ERR_INVALID_ARG      # not 16-byte aligned
    assert call(ws=FAKE + 16) == relay.ERR_INVALID_ARG     # workspace not 256-aligned
    assert lib.relay_kv_append(ctypes.byref(_dims(relay, Hkv=3)), *([ctypes.c_void_p(FAKE)] * 8), 1 << 20,
                               None) == relay.ERR_INVALID_ARG


def test_sys_prefill_host_validation(relay):
    lib = relay.lib()
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    def call(d=None, **o):
        return lib.relay_sys_prefill(ctypes.byref(d or _dims(relay)),
                                     *[vp(o.get(k, FAKE)) for k in ("q", "k", "v", "out", "lse", "ws")],
                                     o.get("ws_bytes", 1 << 20), None)
    assert call(ws=None) == relay.ERR_WORKSPACE
    assert call(d=_dims(relay, D=64)) == relay.ERR_UNSUPPORTED       # tensor-core kernel: D = 128
    assert call(q=None) == relay.ERR_INVALID_ARG
    assert call(out=FAKE + 8) == relay.ERR_INVALID_ARG
    assert call(lse=FAKE + 2) == relay.ERR_INVALID_ARG
    assert call(d=_dims(relay, Ls=0)) == relay.OK                    # nothing to do, nothing queued


def test_rope_host_validation(relay):
    lib = relay.lib()
    vp = lambda x: ctypes.c_void_p(x) if x is not None else None
    call = lambda base=10000.0, **o: lib.relay_rope(ctypes.byref(_dims(relay)),
                                                    *[vp(o.get(k, FAKE)) for k in ("q", "k", "cl", "ql")], base,
                                                    vp(o.get("ws", FAKE)), o.get("ws_bytes", 1 << 20), None)
    assert call(ws=None) == relay.ERR_WORKSPACE
    assert call(base=1.0) == relay.ERR_INVALID_ARG
    assert call(base=float("nan")) == relay.ERR_INVALID_ARG
    assert call(q=None) == relay.ERR_INVALID_ARG
    assert call(k=FAKE + 4) == relay.ERR_INVALID_ARG


def test_fuse_n_host_validation(relay):
    lib = relay.lib()
    arr = lambda *xs: ctypes.cast((ctypes.c_void_p * len(xs))(*xs), ctypes.c_void_p)
    d = _dims(relay)
    ok_parts = arr(FAKE, FAKE)
    assert lib.relay_fuse_n(ctypes.byref(d), 0, ok_parts, ok_parts, None, ctypes.c_void_p(FAKE), None, None) \
        == relay.ERR_INVALID_ARG                                             # K < 1
    assert lib.relay_fuse_n(ctypes.byref(d), 17, ok_parts, ok_parts, None, ctypes.c_void_p(FAKE), None, None) \
        == relay.ERR_INVALID_ARG                                             # K > 16
    assert lib.relay_fuse_n(ctypes.byref(d), 2, arr(FAKE, None), ok_parts, None, ctypes.c_void_p(FAKE), None,
                            None) == relay.ERR_INVALID_ARG                   # a null part
    assert lib.relay_fuse_n(ctypes.byref(d), 2, arr(FAKE, FAKE + 4), ok_parts, None, ctypes.c_void_p(FAKE), None,
                            None) == relay.ERR_INVALID_ARG                   # a misaligned part
    assert lib.relay_fuse_n(ctypes.byref(_dims(relay, B=0)), 2, ok_parts, ok_parts, None, ctypes.c_void_p(FAKE), None,
                            None) == relay.OK                                # nothing to do


def _decode_args(B=2, Lq=1, H=4, Hkv=4, D=64, Ls=32, nb=8, mb=4):
    import torch
    f16, i32 = torch.float16, torch.int32
    return dict(q=torch.zeros(B, Lq, H, D, dtype=f16), sys_k=torch.zeros(Ls, Hkv, D, dtype=f16),
                sys_v=torch.zeros(Ls, Hkv, D, dtype=f16), k_cache=torch.zeros(nb, Hkv, 16, D, dtype=f16),
                v_cache=torch.zeros(nb, Hkv, 16, D, dtype=f16), block_tables=torch.zeros(B, mb, dtype=i32),
                ctx_lens=torch.zeros(B, dtype=i32))


def test_binding_refuses_cpu_tensors(relay):
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        relay.relay_attention_decode(**_decode_args())


def test_binding_checks_shapes(relay):
    """Every tensor the kernels index through the dims is shape-checked before any pointer reaches the
    library (these raise before the CUDA-tensor check, so no device is needed)."""
    import torch
    f16, f32, i32 = torch.float16, torch.float32, torch.int32
    a = _decode_args()
    bad = [
        dict(out=torch.zeros(2, 1, 4, 32, dtype=f16)),                      # out smaller than q
        dict(lse_out=torch.zeros(2, 1, 3, dtype=f32)),
        dict(q_lens=torch.zeros(3, dtype=i32)),
        dict(ctx_lens=torch.zeros(1, dtype=i32)),
        dict(block_tables=torch.zeros(3, 4, dtype=i32)),
        dict(sys_v=torch.zeros(31, 4, 64, dtype=f16)),                      # sys_k / sys_v disagree
        dict(sys_k=torch.zeros(32, 4, 128, dtype=f16), sys_v=torch.zeros(32, 4, 128, dtype=f16)),
        dict(v_cache=torch.zeros(7, 4, 16, 64, dtype=f16)),
        dict(k_cache=torch.zeros(8, 4, 8, 64, dtype=f16), v_cache=torch.zeros(8, 4, 8, 64, dtype=f16)),
    ]
    for over in bad:
        with pytest.raises(ValueError) as e:
            relay.relay_attention_decode(**{**a, **over})
        assert "CUDA" not in str(e.value), (over.keys(), e.value)
    # explicit dims must describe the tensors (sizes and the block-table stride come from them)
    q = a["q"]
    for over in (dict(B=3), dict(Ls=16), dict(num_blocks=9), dict(max_blocks_per_seq=5)):
        d = relay.make_dims(q, 32, 8, 4)
        for k, v in over.items():
            setattr(d, k, v)
        with pytest.raises(ValueError) as e:
            relay._check_dims(d, q, 32, a["k_cache"], a["block_tables"])
        assert "dims" in str(e.value)
    relay._check_dims(relay.make_dims(q, 32, 8, 4), q, 32, a["k_cache"], a["block_tables"])
    # the other entry points
    o = torch.zeros(2, 1, 4, 64, dtype=f32)
    l = torch.zeros(2, 1, 4, dtype=f32)
    with pytest.raises(ValueError, match="o_sys"):
        relay.relay_sys_attn(q, a["sys_k"], a["sys_v"], o_sys=torch.zeros(2, 1, 4, 32, dtype=f32))
    with pytest.raises(ValueError, match="lse_ctx"):
        relay.relay_ctx_attn(q, a["k_cache"], a["v_cache"], a["block_tables"], a["ctx_lens"],
                             lse_ctx=torch.zeros(2, 4, dtype=f32))
    with pytest.raises(ValueError, match="lse_ctx"):
        relay.relay_fuse(o, l, o, torch.zeros(2, 1, 5, dtype=f32))
    with pytest.raises(ValueError, match="o_parts"):
        relay.relay_fuse_n([o, torch.zeros(2, 1, 4, 32, dtype=f32)], [l, l])
    with pytest.raises(ValueError, match="sys_block_ids"):
        relay.relay_baseline_decode(q, a["k_cache"], a["v_cache"], torch.zeros(1, dtype=i32), 32,
                                    a["block_tables"], a["ctx_lens"])
    with pytest.raises(ValueError, match="ctx_lens"):
        relay.relay_kv_append(torch.zeros(2, 1, 4, 64, dtype=f16), torch.zeros(2, 1, 4, 64, dtype=f16),
                              a["block_tables"], torch.zeros(5, dtype=i32), a["k_cache"], a["v_cache"])
    with pytest.raises(ValueError, match="lse_out"):
        relay.relay_sys_prefill(torch.zeros(32, 4, 128, dtype=f16), torch.zeros(32, 4, 128, dtype=f16),
                                torch.zeros(32, 4, 128, dtype=f16), lse_out=torch.zeros(32, 2, dtype=f32))
    with pytest.raises(ValueError, match="k_new"):
        relay.relay_rope(q, a["ctx_lens"], 32, k_new=torch.zeros(2, 2, 4, 64, dtype=f16))


def test_prefixes_host_validation(relay):
    lib = relay.lib()
    d = _dims(relay, Ls=0)
    vp = ctypes.c_void_p
    lens = (ctypes.c_int32 * 3)(2048, 512, 512)
    ptrs = (ctypes.c_void_p * 3)(FAKE, FAKE + 4096, FAKE + 8192)
    assert lib.relay_workspace_size_prefixes(ctypes.byref(d), 3, lens) > 0
    one = lib.relay_workspace_size_prefixes(ctypes.byref(d), 1, lens)
    assert 0 < one < lib.relay_workspace_size_prefixes(ctypes.byref(d), 3, lens)   # more segments, more parts
    for n in (0, 9):
        assert lib.relay_workspace_size_prefixes(ctypes.byref(d), n, lens) == 0
    assert lib.relay_workspace_size_prefixes(ctypes.byref(d), 2, (ctypes.c_int32 * 2)(5, -1)) == 0

    def call(n=3, k=ptrs, v=ptrs, L=lens, mask=None, q=FAKE, dims=d, B0=False):
        dd = _dims(relay, Ls=0, B=0) if B0 else dims
        return lib.relay_attention_decode_prefixes(ctypes.byref(dd), vp(q), n, k, v, L, vp(mask) if mask else None,
                                                   vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, vp(FAKE), None,
                                                   vp(FAKE), 1 << 30, None)
    assert call(n=0) == relay.ERR_INVALID_ARG
    assert call(n=9) == relay.ERR_INVALID_ARG
    assert call(L=(ctypes.c_int32 * 3)(10, -1, 3)) == relay.ERR_INVALID_ARG
    assert call(k=(ctypes.c_void_p * 3)(FAKE, None, FAKE)) == relay.ERR_INVALID_ARG        # segment 1 has keys
    assert call(k=(ctypes.c_void_p * 3)(FAKE, FAKE + 8, FAKE)) == relay.ERR_INVALID_ARG    # not 16-byte aligned
    assert call(mask=FAKE + 2) == relay.ERR_INVALID_ARG                                    # mask not 4-byte aligned
    assert call(q=None) == relay.ERR_INVALID_ARG
    # an empty segment may have no pointers; with nothing to do, nothing is queued
    assert call(k=(ctypes.c_void_p * 3)(FAKE, FAKE, FAKE), L=(ctypes.c_int32 * 3)(64, 0, 64), B0=True) == relay.OK
