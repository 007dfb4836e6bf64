"""Shared helpers of the GPU parity tests: move a synth.Case to the device,
call the library through its binding, and compare with the oracle under the
stated tolerance."""
import math

import numpy as np
import torch

import oracle
import shared_prompt_decode_gb300 as relay
import synth

# fp16 I/O, fp32 accumulation: max-abs 2e-3 and normwise relative 1e-2 on the
# outputs; 1e-3 absolute on the natural-log LSE.
ATOL = 2e-3
NORM_RTOL = 1e-2
LSE_ATOL = 1e-3

DEV = torch.device("cuda:0")


def to_dev(case):
    g = {k: getattr(case, k).to(DEV) for k in ("q", "sys_k", "sys_v", "k_cache", "v_cache",
                                              "block_tables", "ctx_lens")}
    g["q_lens"] = None if case.q_lens is None else case.q_lens.to(DEV)
    return g


def _mq(case):
    return case.total_q() if case.q_lens is not None else 0


def run_fused(case, ws=None, ctx_split=0, sys_range=0, g=None):
    g = g or to_dev(case)
    lse = torch.full((case.B, case.Lq, case.H), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.full_like(g["q"], float("nan"))
    relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"], g["block_tables"],
                                 g["ctx_lens"], g["q_lens"], out=out, lse_out=lse, workspace=ws,
                                 max_q_total=_mq(case), ctx_split=ctx_split, sys_range=sys_range)
    torch.cuda.synchronize()
    return out, lse


def run_split(case, ctx_split=0, sys_range=0):
    g = to_dev(case)
    o_s, l_s = relay.relay_sys_attn(g["q"], g["sys_k"], g["sys_v"], g["q_lens"], max_q_total=_mq(case),
                                    sys_range=sys_range)
    o_c, l_c = relay.relay_ctx_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["ctx_lens"],
                                    g["q_lens"], max_q_total=_mq(case), ctx_split=ctx_split)
    lse = torch.full((case.B, case.Lq, case.H), float("nan"), dtype=torch.float32, device=DEV)
    out = relay.relay_fuse(o_s, l_s, o_c, l_c, g["q_lens"], lse_out=lse)
    torch.cuda.synchronize()
    return o_s, l_s, o_c, l_c, out, lse


def run_baseline(case, ctx_split=0):
    kp, vp, ids = synth.with_system_in_pool(case)
    g = to_dev(case)
    lse = torch.full((case.B, case.Lq, case.H), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.full_like(g["q"], float("nan"))
    relay.relay_baseline_decode(g["q"], kp.to(DEV), vp.to(DEV), ids.to(DEV), case.Ls, g["block_tables"],
                                g["ctx_lens"], g["q_lens"], out=out, lse_out=lse, max_q_total=_mq(case),
                                ctx_split=ctx_split)
    torch.cuda.synchronize()
    return out, lse


def valid_mask(case):
    m = np.zeros((case.B, case.Lq), dtype=bool)
    for b, n in enumerate(case.q_lens_list()):
        m[b, :n] = True
    return m


def check(got, ref, what="out", mask=None):
    """Compare a device result with oracle values on the valid rows."""
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if mask is not None:
        g, r = g[mask], r[mask]
    assert g.shape == r.shape
    fin = np.isfinite(r)
    assert np.array_equal(g[~fin], r[~fin]), f"{what}: non-finite entries differ"
    assert np.all(np.isfinite(g[fin])), f"{what}: non-finite value where the oracle is finite"
    g, r = g[fin], r[fin]
    if r.size == 0:
        return 0.0
    err = np.abs(g - r)
    amax = float(err.max())
    if what.startswith("lse"):
        assert amax <= LSE_ATOL, f"{what}: max abs err {amax:.3e}"
        return amax
    norm = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert amax <= ATOL, f"{what}: max abs err {amax:.3e} (normwise {norm:.3e})"
    assert norm <= NORM_RTOL, f"{what}: normwise rel err {norm:.3e}"
    return amax


def check_full(case, out, lse, part="full"):
    ref, ref_lse = oracle.attention_full(case, part)
    m = valid_mask(case)
    check(out, ref, "out", m)
    check(lse, ref_lse, "lse", m)


def check_rows(case, out, lse, rows, part="full"):
    ref, ref_lse = oracle.attention_rows(case, rows, part)
    idx = tuple(np.array(rows).T)
    o = out.double().cpu().numpy()[idx]
    l = lse.double().cpu().numpy()[idx]
    check(o, ref, "out")
    check(l, ref_lse, "lse")
