"""Failure detection in the tensor-core system step: every wait of its
warp-specialised pipeline is bounded in time, and a wait that gives up must
end the kernel cleanly -- copies and MMAs in flight drained, TMEM freed, the
call returning -- and report RELAY_FLAG_WAIT_TIMEOUT instead of hanging.

The wait never runs out in a correct run, so the test uses a build of the
same sources whose protocol limit is 0 ns (RELAY_WAIT_LIMIT_NS=0): the first
wait that is not met at once gives up.  Draining stays bounded by 1 s in
that build too.  No fault, trap or endless loop is involved.  Afterwards the
normal library, in the same CUDA context, must still match the oracle."""
import ctypes

import pytest
import torch

import synth
from tests import relay_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    from shared_prompt_decode_gb300 import build
    import shared_prompt_decode_gb300 as relay
    build.build()
    path = build.build(variant="wait0", defines=["RELAY_WAIT_LIMIT_NS=0ull"])
    short = ctypes.CDLL(path)
    short.relay_attention_decode.restype = ctypes.c_int
    short.relay_attention_decode.argtypes = [ctypes.POINTER(relay.Dims)] + [ctypes.c_void_p] * 11 + \
        [ctypes.c_size_t, ctypes.c_void_p]
    short.relay_device_status.restype = ctypes.c_int
    short.relay_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_void_p]
    return relay, short


def _case():
    # 5 requests x 64 query rows = 320 rows per head (> 256): the system step runs on the tcgen05 kernel
    w = synth.Workload("timeout_tc", B=5, H=2, D=128, Ls=1024, ctx_dist=("uniform", 64, 96), value_scale=0.5, Lq=64)
    return synth.make_case(w, seed=3)


def test_wait_that_gives_up_is_reported_and_leaves_the_context_usable(libs):
    relay, short = libs
    case = _case()
    g = T.to_dev(case)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
    ws = relay.make_workspace(dims)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    seen = 0
    for _ in range(3):
        out = torch.zeros_like(g["q"])
        rc = short.relay_attention_decode(ctypes.byref(dims), p(g["q"]), p(g["sys_k"]), p(g["sys_v"]),
                                          p(g["k_cache"]), p(g["v_cache"]), p(g["block_tables"]),
                                          p(g["ctx_lens"]), None, p(out), None, p(ws), ws.numel(), stream)
        assert rc == relay.OK, relay.status_string(rc)
        torch.cuda.synchronize()                       # the call returned and the kernels ended
        flags = ctypes.c_uint32(0)
        short.relay_device_status(p(ws), ctypes.byref(flags), stream)
        seen |= flags.value
    assert seen & relay.FLAG_WAIT_TIMEOUT
    assert seen & ~relay.FLAG_WAIT_TIMEOUT == 0        # no other check fired
    # the same context, the normal library: correct results, no flag
    out, lse = T.run_fused(case, ws=ws, g=g)
    assert relay.device_status(ws) == 0
    T.check_full(case, out, lse)
