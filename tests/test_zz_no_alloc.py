"""relay_attention_decode_noalloc: the entry point for callers that cannot
allocate device memory when they call (a serving process whose allocator owns
all device memory, or a decode loop that must not reach cudaMalloc).  It runs
the same computation with its scratch in a fixed buffer inside the library.

Called through the C ABI and checked, on two calls in a row (every call
reuses the same buffer), against the fp64 oracle and against
relay_attention_decode (which uses a caller-allocated workspace) within the
parity tolerance.  The device-side check flags of the shared buffer are read
back with relay_noalloc_device_status.  This file is collected last so that a
run stopping at the first failure has run everything else."""
import ctypes

import pytest
import torch

import synth
from tests import relay_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def relay():
    from shared_prompt_decode_gb300 import build
    build.build()
    import shared_prompt_decode_gb300 as r
    lib = r.lib()
    fn = lib.relay_attention_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(r.Dims)] + [ctypes.c_void_p] * 11
    st = lib.relay_noalloc_device_status
    st.restype = ctypes.c_int
    st.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    return r


def _status(relay):
    flags = ctypes.c_uint32(0)
    rc = relay.lib().relay_noalloc_device_status(ctypes.byref(flags),
                                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc in (relay.OK, relay.ERR_DEVICE_CHECK), relay.status_string(rc)
    assert (rc == relay.OK) == (flags.value == 0)
    return flags.value


def _noalloc(relay, dims, g, out, lse):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return relay.lib().relay_attention_decode_noalloc(
        ctypes.byref(dims), p(g["q"]), p(g["sys_k"]), p(g["sys_v"]), p(g["k_cache"]), p(g["v_cache"]),
        p(g["block_tables"]), p(g["ctx_lens"]), p(g["q_lens"]), p(out), p(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,seed", [("llama2_7b", 21), ("tiny", 22)])
def test_noalloc_matches_workspace_entry_point(relay, name, seed):
    case = synth.make_case(name, seed)
    g = T.to_dev(case)
    ref_out, ref_lse = T.run_fused(case, g=g)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
    assert relay.workspace_size(dims) <= (32 << 20)
    for call in range(2):                   # the shared buffer keeps the previous call's contents
        out = torch.full_like(g["q"], float("nan"))
        lse = torch.full((case.B, case.Lq, case.H), float("nan"), dtype=torch.float32, device=T.DEV)
        rc = _noalloc(relay, dims, g, out, lse)
        assert rc == relay.OK, relay.status_string(rc)
        torch.cuda.synchronize()
        assert _status(relay) == 0
        T.check(out, ref_out.double().cpu().numpy(), f"out (call {call})")
        T.check(lse, ref_lse.double().cpu().numpy(), f"lse (call {call})")
        T.check_full(case, out, lse)


def test_noalloc_device_status_reports_a_bad_block(relay):
    case = synth.make_case("tiny", 23)
    g = T.to_dev(case)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
    bad = dict(g, block_tables=g["block_tables"].clone())
    bad["block_tables"][2, 0] = case.num_blocks + 7           # outside the pool: skipped and flagged
    out = torch.zeros_like(g["q"])
    assert _noalloc(relay, dims, bad, out, None) == relay.OK
    assert _status(relay) & relay.FLAG_BAD_BLOCK
    assert _status(relay) == 0                                # reading clears the flags
    # the next clean call is correct and raises nothing
    lse = torch.full((case.B, case.Lq, case.H), float("nan"), dtype=torch.float32, device=T.DEV)
    assert _noalloc(relay, dims, g, out, lse) == relay.OK
    assert _status(relay) == 0
    T.check_full(case, out, lse)


def test_noalloc_rejects_oversized_shapes(relay):
    # a batch whose workspace would exceed the fixed buffer: rejected on the host
    dims = relay.Dims(256, 1, 32, 128, 4096, 16, 40000, 128, 0, 0, 0, 0.0)
    assert relay.workspace_size(dims) > (32 << 20)
    g = {k: None for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache", "block_tables", "ctx_lens", "q_lens")}
    dummy = torch.empty(16, dtype=torch.float16, device=T.DEV)
    for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache"):
        g[k] = dummy
    g["block_tables"] = g["ctx_lens"] = torch.empty(16, dtype=torch.int32, device=T.DEV)
    assert _noalloc(relay, dims, g, dummy, None) == relay.ERR_WORKSPACE
