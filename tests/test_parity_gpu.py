"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Tolerance (fp16 I/O, fp32 accumulation): max-abs 2e-3 and normwise relative
1e-2 on outputs, 1e-3 absolute on the natural-log LSE.  Page-table indexing
is checked bit for bit (one-hot keys, pool relabelling).  Unused pool slots
and padding query rows are NaN, so an unmasked read fails the comparison.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import relay_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from shared_prompt_decode_gb300 import build
    build.build()
    oracle.build()
    assert torch.cuda.is_available()


def wl(name, **kw):
    return synth.workload(name, **kw)


# ----------------------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fused(seed):
    case = synth.make_case("tiny", seed)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


def test_tiny_three_steps():
    case = synth.make_case("tiny", 4)
    o_s, l_s, o_c, l_c, out, lse = T.run_split(case)
    ref_s, refl_s = oracle.attention_full(case, "sys")
    ref_c, refl_c = oracle.attention_full(case, "ctx")
    m = T.valid_mask(case)
    T.check(o_s, ref_s, "o_sys", m)
    T.check(l_s, refl_s, "lse_sys", m)
    T.check(o_c, ref_c, "o_ctx", m)
    T.check(l_c, refl_c, "lse_ctx", m)
    T.check_full(case, out, lse)


@pytest.mark.parametrize("seed", [0, 1])
def test_llama2_7b_full(seed):
    case = synth.make_case("llama2_7b", seed)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


def test_llama2_7b_three_steps():
    case = synth.make_case("llama2_7b", 2)
    o_s, l_s, o_c, l_c, out, lse = T.run_split(case)
    m = T.valid_mask(case)
    ref_s, refl_s = oracle.attention_full(case, "sys")
    T.check(o_s, ref_s, "o_sys", m)
    T.check(l_s, refl_s, "lse_sys", m)
    ref_c, refl_c = oracle.attention_full(case, "ctx")
    T.check(o_c, ref_c, "o_ctx", m)
    T.check(l_c, refl_c, "lse_ctx", m)
    T.check_full(case, out, lse)


# every (request, row, head) of every system-prompt length, 512 .. 16384
@pytest.mark.parametrize("Ls", synth.SWEEP_LS)
def test_llama30b_sweep(Ls):
    case = synth.make_case(wl("llama30b_sweep", Ls=Ls), 0)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


# every (request, row, head) of the batch-256 workload
def test_llama2_7b_b256():
    case = synth.make_case("llama2_7b_b256", 0)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


# Rows of the 13B mixed workload checked against the oracle (7,360 of its
# 43,200 (request, row, head) outputs): the one row of every decode request
# (0..55) on every head, and every row of every chunk request (56..63) on
# five heads spread over the 40 (0, 9, 19, 29, 39).  Every output is also
# checked to be finite, and every padding row untouched.
def mixed_rows(case):
    ql = case.q_lens_list()
    rows = [(b, 0, h) for b in range(case.B) if ql[b] == 1 for h in range(case.H)]
    rows += [(b, i, h) for b in range(case.B) if ql[b] > 1 for i in range(ql[b]) for h in (0, 9, 19, 29, 39)]
    return rows


def test_llama2_13b_mixed():
    case = synth.make_case("llama2_13b_mixed", 0)
    out, lse = T.run_fused(case)
    rows = mixed_rows(case)
    assert len(rows) == 56 * 40 + 8 * 128 * 5
    T.check_rows(case, out, lse, rows)
    # outputs are finite everywhere they are defined, and padding rows untouched
    ql = case.q_lens_list()
    o = out.float().cpu()
    for b in range(case.B):
        assert torch.isfinite(o[b, :ql[b]]).all()
        assert torch.isnan(o[b, ql[b]:]).all()


# ----------------------------------------------------------------------------- merge paths
@pytest.mark.parametrize("ctx_split,sys_range", [(64, 64), (128, 192), (64, 0), (0, 64)])
def test_forced_splits_tiny(ctx_split, sys_range):
    case = synth.make_case("tiny", 5)
    out, lse = T.run_fused(case, ctx_split=ctx_split, sys_range=sys_range)
    T.check_full(case, out, lse)
    o_s, l_s, o_c, l_c, out2, lse2 = T.run_split(case, ctx_split=ctx_split, sys_range=sys_range)
    T.check_full(case, out2, lse2)


def test_forced_splits_llama2_7b():
    case = synth.make_case("llama2_7b", 3)
    out, lse = T.run_fused(case, ctx_split=128, sys_range=256)
    T.check_full(case, out, lse)


# ----------------------------------------------------------------------------- edge cases
EDGE = [
    ("empty_ctx_some", dict(), [0, 5, 0, 17], None),
    ("empty_system", dict(Ls=0), None, None),
    ("both_empty_some", dict(Ls=0), [0, 0, 4, 0], None),
    ("ragged_block_edges", dict(), [1, 15, 16, 17], None),
    ("ragged_tile_edges", dict(), [63, 64, 65, 128], None),
    ("short_system", dict(Ls=1), [3, 64, 33, 0], None),
    ("odd_system", dict(Ls=100), [100, 1, 2, 64], None),
    ("single_request", dict(B=1), [37], None),
]


@pytest.mark.parametrize("name,over,ctx,ql", EDGE, ids=[e[0] for e in EDGE])
def test_edge_cases(name, over, ctx, ql):
    case = synth.make_case(wl("tiny", pool_blocks=40, **over), 6, ctx_lens=ctx, q_lens=ql)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)
    *_, out2, lse2 = T.run_split(case)
    T.check_full(case, out2, lse2)
    outb, lseb = T.run_baseline(case)
    T.check_full(case, outb, lseb)


@pytest.mark.parametrize("D", [64, 128])
def test_mixed_query_rows(D):
    w = synth.Workload("mixed", B=5, H=3, D=D, Ls=300, ctx_dist=("uniform", 1, 200), value_scale=0.5, Lq=80)
    case = synth.make_case(w, 7, ctx_lens=[150, 80, 5, 200, 2], q_lens=[1, 80, 0, 65, 3])
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)
    *_, out2, lse2 = T.run_split(case, ctx_split=64)
    T.check_full(case, out2, lse2)
    outb, lseb = T.run_baseline(case)
    T.check_full(case, outb, lseb)
    # rows past q_lens are untouched
    assert torch.isnan(out[2].float()).all() and torch.isnan(out[0, 1:].float()).all()


def test_max_batch():
    w = synth.Workload("maxb", B=512, H=2, D=64, Ls=64, ctx_dist=("uniform", 0, 40), value_scale=1.0)
    case = synth.make_case(w, 8)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


# ----------------------------------------------------------------------------- non-relay baseline
@pytest.mark.parametrize("name,rows", [("tiny", None), ("llama2_7b", 600)])
def test_baseline(name, rows):
    case = synth.make_case(name, 9)
    out, lse = T.run_baseline(case)
    if rows is None:
        T.check_full(case, out, lse)
    else:
        T.check_rows(case, out, lse, synth.sample_rows(case, rows, seed=3))


# ----------------------------------------------------------------------------- page-table indexing, bit-exact
def _one_hot_ctx(case, hot):
    """Zero every real key; make key hot[(b,h)] of each pair dominate."""
    kc = case.k_cache.clone()
    kc = torch.where(torch.isnan(kc), kc, torch.zeros_like(kc))
    sk = torch.zeros_like(case.sys_k)
    D = case.D
    expect = torch.empty(case.B, case.H, D, dtype=torch.float16)
    for (b, h), t in hot.items():
        blk, slot = int(case.block_tables[b, t // 16]), t % 16
        qv = case.q[b, 0, h].double()
        kc[blk, h, slot] = (8.0 * qv / qv.norm() * math.sqrt(D)).to(torch.float16)
        expect[b, h] = case.v_cache[blk, h, slot]
    c = synth.Case(case.wl, case.seed, case.q, sk, case.sys_v, kc, case.v_cache, case.block_tables,
                   case.ctx_lens, case.q_lens)
    return c, expect


def test_one_hot_every_context_position_tiny():
    case = synth.make_case("tiny", 10)
    n = [int(x) for x in case.ctx_lens]
    for r in range(max(n)):
        hot = {(b, h): (r + 7 * h) % n[b] for b in range(case.B) for h in range(case.H)}
        c, expect = _one_hot_ctx(case, hot)
        out, _ = T.run_fused(c)
        assert torch.equal(out[:, 0].cpu(), expect), f"position sweep step {r}"


def test_one_hot_context_llama2_7b():
    case = synth.make_case("llama2_7b", 11)
    g = torch.Generator().manual_seed(0)
    for r in range(3):
        hot = {(b, h): int(torch.randint(0, int(case.ctx_lens[b]), (1,), generator=g))
               for b in range(case.B) for h in range(case.H)}
        c, expect = _one_hot_ctx(case, hot)
        out, _ = T.run_fused(c)
        assert torch.equal(out[:, 0].cpu(), expect)
        outb, _ = T.run_baseline(c)
        assert torch.equal(outb[:, 0].cpu(), expect)


def test_one_hot_system_position():
    case = synth.make_case("llama2_7b", 12)
    q = case.q.clone()
    q[:] = q[0:1]                         # one query per head, shared by every request
    kc = torch.where(torch.isnan(case.k_cache), case.k_cache, torch.zeros_like(case.k_cache))
    sk = torch.zeros_like(case.sys_k)
    expect = torch.empty(case.H, case.D, dtype=torch.float16)
    for h in range(case.H):
        s = (h * 61 + 5) % case.Ls
        qv = q[0, 0, h].double()
        sk[s, h] = (8.0 * qv / qv.norm() * math.sqrt(case.D)).to(torch.float16)
        expect[h] = case.sys_v[s, h]
    c = synth.Case(case.wl, case.seed, q, sk, case.sys_v, kc, case.v_cache, case.block_tables,
                   case.ctx_lens, case.q_lens)
    out, _ = T.run_fused(c)
    assert torch.equal(out[:, 0].cpu(), expect[None].expand(case.B, -1, -1))


def test_pool_relabelling_bitwise():
    case = synth.make_case("llama2_7b", 13)
    out1, lse1 = T.run_fused(case)
    out2, lse2 = T.run_fused(synth.relabel_pool(case, 77))
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


# ----------------------------------------------------------------------------- runtime behaviour
def test_deterministic_and_workspace_reuse():
    import shared_prompt_decode_gb300 as relay
    case = synth.make_case("llama2_7b", 14)
    g = T.to_dev(case)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
    ws = relay.make_workspace(dims)
    outs = [T.run_fused(case, ws=ws, g=g) for _ in range(3)]
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    # the same workspace serves the three-step path in between
    relay.relay_sys_attn(g["q"], g["sys_k"], g["sys_v"], workspace=ws)
    o4, l4 = T.run_fused(case, ws=ws, g=g)
    assert torch.equal(o4, outs[0][0])
    assert relay.device_status(ws) == 0


def test_cuda_graph_replay():
    import shared_prompt_decode_gb300 as relay
    case = synth.make_case("llama2_7b", 15)
    g = T.to_dev(case)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, Hkv=case.Hkv)
    ws = relay.make_workspace(dims)
    out = torch.empty_like(g["q"])
    ref, _ = T.run_fused(case, g=g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"],
                                     g["block_tables"], g["ctx_lens"], out=out, workspace=ws, dims=dims)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"],
                                     g["block_tables"], g["ctx_lens"], out=out, workspace=ws, dims=dims)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


@pytest.mark.parametrize("what", ["block", "ctx_len", "q_len", "q_total"])
def test_device_checks_flag_bad_values(what):
    import shared_prompt_decode_gb300 as relay
    case = synth.make_case(wl("tiny", Lq=2), 16, q_lens=[1, 2, 1, 2])
    g = T.to_dev(case)
    mq = case.total_q()
    expect = {"block": relay.FLAG_BAD_BLOCK, "ctx_len": relay.FLAG_BAD_CTX_LEN,
              "q_len": relay.FLAG_BAD_Q_LEN, "q_total": relay.FLAG_Q_TOTAL}[what]
    if what == "block":
        g["block_tables"][1, 0] = case.num_blocks + 3
    elif what == "ctx_len":
        g["ctx_lens"][2] = case.max_blocks * 16 + 1
    elif what == "q_len":
        g["q_lens"][0] = 3
    else:
        mq = 3
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, max_q_total=mq)
    ws = relay.make_workspace(dims)
    out = torch.zeros_like(g["q"])
    relay.relay_attention_decode(g["q"], g["sys_k"], g["sys_v"], g["k_cache"], g["v_cache"],
                                 g["block_tables"], g["ctx_lens"], g["q_lens"], out=out, workspace=ws, dims=dims)
    assert relay.device_status(ws) & expect
    assert relay.device_status(ws) == 0        # reading clears the flags
    # the workspace stays usable: a clean call afterwards is correct
    case2 = synth.make_case(wl("tiny", Lq=2), 17, q_lens=[1, 2, 1, 2])
    dims2 = relay.make_dims(g["q"], case2.Ls, case2.num_blocks, case2.max_blocks, max_q_total=case2.total_q())
    ws2 = ws if relay.workspace_size(dims2) <= ws.numel() else relay.make_workspace(dims2)
    out2, lse2 = T.run_fused(case2, ws=ws2)
    T.check_full(case2, out2, lse2)


# ----------------------------------------------------------------------------- tensor-core system step
# Batches with more than 256 query rows per head run the system step on the
# tcgen05 kernel (pairs of 128-row tiles, 128-key stages, one S buffer that
# the two tiles take in turn); ragged rows and keys on purpose, a lone tile
# beside a pair (257 rows), and ranges of 1 and 2 stages, which take the
# pipeline's prologue-only and shortest-loop paths.
TC_CASES = [
    ("rows257_keys1000", 257, 1, 1000, None),
    ("rows300_keys64", 300, 1, 64, None),
    ("rows300_keys100", 300, 1, 100, None),
    ("rows513_keys150", 171, 3, 150, None),
    ("rows600_keys4097", 150, 4, 4097, None),
    ("chunks_qlens", 6, 128, 700, [128, 1, 77, 128, 3, 90]),
]


@pytest.mark.parametrize("name,B,Lq,Ls,ql", TC_CASES, ids=[c[0] for c in TC_CASES])
def test_tensor_core_system_step(name, B, Lq, Ls, ql):
    w = synth.Workload(name, B=B, H=3, D=128, Ls=Ls, ctx_dist=("uniform", 0, 48), value_scale=0.5, Lq=Lq)
    case = synth.make_case(w, 31, q_lens=ql)
    if ql is not None:
        case.ctx_lens[:] = torch.maximum(case.ctx_lens, case.q_lens)
        case = synth.make_case(w, 31, ctx_lens=[int(x) for x in case.ctx_lens], q_lens=ql)
    assert case.total_q() > 256
    o_s, l_s, o_c, l_c, out2, lse2 = T.run_split(case)
    ref_s, refl_s = oracle.attention_full(case, "sys")
    m = T.valid_mask(case)
    T.check(o_s, ref_s, "o_sys", m)
    T.check(l_s, refl_s, "lse_sys", m)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)
    T.check_full(case, out2, lse2)


# ----------------------------------------------------------------------------- chunk rows' own contexts on tcgen05
# Requests of Lq * G >= 64 virtual rows per KV head take their own context on
# the tensor-core kernel, in the grid of the system step: paged copies (four
# 16-token page boxes per 128-key stage), a causal limit per row, and the V
# slots past the context zeroed (the pool's unused slots hold NaN).  Long and
# ragged contexts, two tile pairs of one request (300 rows), contexts shorter
# than the chunk (rows that see no context key), one-row and empty requests
# beside them, grouped-query heads, and every request at Lq rows (no q_lens).
CTX_TC_CASES = [
    ("mha_pairs", dict(B=6, H=2, Lq=300, Ls=200), [300, 1, 129, 64, 0, 2], [1500, 700, 129, 3000, 50, 1]),
    ("gqa", dict(B=4, H=8, Hkv=2, Lq=40, Ls=130), [40, 1, 17, 33], [2000, 300, 17, 999]),
    ("all_rows", dict(B=3, H=2, Lq=64, Ls=64), None, [64, 1000, 333]),
]


@pytest.mark.parametrize("name,over,ql,ctx", CTX_TC_CASES, ids=[c[0] for c in CTX_TC_CASES])
def test_chunk_context_on_tensor_cores(name, over, ql, ctx):
    w = synth.Workload(name, D=128, ctx_dist=("uniform", 1, 2), value_scale=0.5, **over)
    case = synth.make_case(w, 37, ctx_lens=ctx, q_lens=ql)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)
    *_, out2, lse2 = T.run_split(case)
    T.check_full(case, out2, lse2)


def test_mixed_batch_few_decode_requests():
    # prompt chunks on the tensor cores (system step and their own contexts)
    # with only four decode requests streaming beside them: the grid yields
    # only the SMs those requests need; every output against the oracle
    w = synth.Workload("mixed_few_decode", B=12, H=8, D=128, Ls=4096, ctx_dist=("uniform", 1, 2048),
                       value_scale=0.5, Lq=128, chunk_requests=8)
    case = synth.make_case(w, 43)
    assert case.total_q() > 256
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


def test_chunk_context_bad_block_is_flagged():
    # a page id outside the pool in a chunk request's context: read as zeros
    # and flagged; the next clean call in the same workspace is exact
    import shared_prompt_decode_gb300 as relay
    w = synth.Workload("ctx_bad", B=3, H=2, D=128, Ls=64, ctx_dist=("uniform", 1, 2), value_scale=0.5, Lq=64)
    case = synth.make_case(w, 41, ctx_lens=[100, 1, 200], q_lens=[64, 1, 64])
    g = T.to_dev(case)
    dims = relay.make_dims(g["q"], case.Ls, case.num_blocks, case.max_blocks, max_q_total=case.total_q())
    ws = relay.make_workspace(dims)
    bad = dict(g, block_tables=g["block_tables"].clone())
    bad["block_tables"][2, 3] = case.num_blocks + 5
    out = torch.zeros_like(g["q"])
    relay.relay_attention_decode(bad["q"], bad["sys_k"], bad["sys_v"], bad["k_cache"], bad["v_cache"],
                                 bad["block_tables"], bad["ctx_lens"], bad["q_lens"], out=out, workspace=ws,
                                 dims=dims)
    assert relay.device_status(ws) & relay.FLAG_BAD_BLOCK
    out, lse = T.run_fused(case, ws=ws, g=g)
    assert relay.device_status(ws) == 0
    T.check_full(case, out, lse)


# ----------------------------------------------------------------------------- grouped-query heads
# Hkv KV heads serve H query heads (query head h reads KV head h / (H / Hkv)):
# every path -- one call, the three separate steps, the non-relay baseline,
# multi-row requests, and the tensor-core system step -- against the oracle.
GQA_CASES = [
    ("tiny_gqa", {}),
    ("tiny_mqa", {}),
    ("tiny_gqa", dict(Lq=3, chunk_requests=2)),
    ("llama2_70b_gqa", {}),
]


@pytest.mark.parametrize("name,over", GQA_CASES, ids=["gqa", "mqa", "gqa_chunks", "llama2_70b_gqa"])
def test_grouped_query_heads(name, over):
    case = synth.make_case(synth.workload(name, **over), 21)
    assert case.Hkv < case.H
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)
    o_s, l_s, o_c, l_c, out2, lse2 = T.run_split(case)
    m = T.valid_mask(case)
    ref_s, refl_s = oracle.attention_full(case, "sys")
    T.check(o_s, ref_s, "o_sys", m)
    T.check(l_s, refl_s, "lse_sys", m)
    T.check_full(case, out2, lse2)
    outb, lseb = T.run_baseline(case)
    T.check_full(case, outb, lseb)


# The system step runs over virtual rows (query row, query head of the group)
# of each KV head: 300 rows x 2 heads, and 48 decode rows x 8 heads of one KV
# head, where only the grouping takes it past 256 rows onto the tensor cores.
@pytest.mark.parametrize("B,Lq,H,Hkv", [(150, 2, 4, 2), (48, 1, 8, 1)], ids=["rows300_g2", "rows48_mqa8"])
def test_grouped_query_heads_tensor_core_system_step(B, Lq, H, Hkv):
    w = synth.Workload("tc_gqa", B=B, H=H, D=128, Ls=1000, ctx_dist=("uniform", 0, 48), value_scale=0.5,
                       Lq=Lq, Hkv=Hkv)
    case = synth.make_case(w, 23)
    assert case.total_q() * (H // Hkv) > 256
    o_s, l_s, o_c, l_c, out2, lse2 = T.run_split(case)
    m = T.valid_mask(case)
    ref_s, refl_s = oracle.attention_full(case, "sys")
    T.check(o_s, ref_s, "o_sys", m)
    T.check(l_s, refl_s, "lse_sys", m)
    out, lse = T.run_fused(case)
    T.check_full(case, out, lse)


# ----------------------------------------------------------------------------- KV append
# relay_kv_append must leave the pools bit-identical to the oracle's append
# (every slot: the written rows, and the untouched and NaN slots as they were).
def _kv_append_case(name, over, seed):
    case = synth.make_case(synth.workload(name, **over), seed)
    g = torch.Generator().manual_seed(seed + 100)
    shape = (case.B, case.Lq, case.Hkv, case.D)
    return case, torch.randn(*shape, generator=g).half(), torch.randn(*shape, generator=g).half()


@pytest.mark.parametrize("name,over", [("tiny", {}), ("tiny_gqa", dict(Lq=3, chunk_requests=2)),
                                        ("llama2_7b", {}), ("llama2_13b_mixed", dict(Ls=64))],
                         ids=["tiny", "gqa_chunks", "llama2_7b", "13b_mixed_chunks"])
def test_kv_append_bit_exact(name, over):
    import shared_prompt_decode_gb300 as relay
    case, k_new, v_new = _kv_append_case(name, over, 41)
    ref_k, ref_v = oracle.kv_append(case, k_new, v_new)
    g = T.to_dev(case)
    kc, vc = g["k_cache"].clone(), g["v_cache"].clone()
    ws = relay.relay_kv_append(k_new.to(T.DEV), v_new.to(T.DEV), g["block_tables"], g["ctx_lens"], kc, vc,
                               q_lens=g["q_lens"])
    torch.cuda.synchronize()
    assert relay.device_status(ws) == 0
    assert torch.equal(kc.cpu().view(torch.int16), ref_k.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), ref_v.view(torch.int16))


def test_kv_append_device_checks():
    import shared_prompt_decode_gb300 as relay
    case, k_new, v_new = _kv_append_case("tiny", dict(Lq=2, chunk_requests=4), 43)
    g = T.to_dev(case)
    bt = g["block_tables"].clone()
    bt[0, :] = case.num_blocks + 5                  # request 0: every block id out of range
    cl = g["ctx_lens"].clone()
    cl[1] = 1                                       # request 1: 2 new rows, 1-token context
    kc, vc = g["k_cache"].clone(), g["v_cache"].clone()
    ws = relay.relay_kv_append(k_new.to(T.DEV), v_new.to(T.DEV), bt, cl, kc, vc, q_lens=g["q_lens"])
    flags = relay.device_status(ws)
    assert flags & relay.FLAG_BAD_BLOCK and flags & relay.FLAG_BAD_CTX_LEN
    # the valid requests (2, 3) are written exactly as the oracle writes them
    from dataclasses import replace
    sub = replace(case, q_lens=torch.tensor([0, 0, 2, 2], dtype=torch.int32))
    ref_k, _ = oracle.kv_append(sub, k_new, v_new)
    assert torch.equal(kc.cpu().view(torch.int16), ref_k.view(torch.int16))


# ----------------------------------------------------------------------------- system-prompt prefill
# relay_sys_prefill (tcgen05 kernel, causal) against the oracle: every row for
# short prompts; first, last, diagonal-tile and random rows for a 32768-token
# prompt at the Llama-2-13B shape.
PREFILL_CASES = [
    (300, 4, 2, None), (2048, 32, 32, None), (1000, 8, 1, None), (129, 2, 2, None),
    (32768, 40, 40, 192), (1, 2, 2, None), (64, 3, 1, None), (200, 8, 2, None),
]


@pytest.mark.parametrize("Ls,H,Hkv,sample", PREFILL_CASES,
                         ids=["Ls300_gqa", "Ls2048_llama2_7b", "Ls1000_mqa", "Ls129_ragged", "Ls32768_13b_sampled",
                              "Ls1_single_key", "Ls64_one_partial_tile", "Ls200_group4"])
def test_sys_prefill(Ls, H, Hkv, sample):
    import shared_prompt_decode_gb300 as relay
    g = torch.Generator().manual_seed(Ls + H)
    q = (torch.randn(Ls, H, 128, generator=g) * 0.5).half()
    k = (torch.randn(Ls, Hkv, 128, generator=g) * 0.5).half()
    v = (torch.randn(Ls, Hkv, 128, generator=g) * 0.5).half()
    lse = torch.full((Ls, H), float("nan"), dtype=torch.float32, device=T.DEV)
    ws = torch.zeros(256, dtype=torch.uint8, device=T.DEV)
    out = relay.relay_sys_prefill(q.to(T.DEV), k.to(T.DEV), v.to(T.DEV), lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    assert relay.device_status(ws) == 0
    if sample is None:
        rows = [(t, h) for t in range(Ls) for h in range(H)]
    else:
        gen = torch.Generator().manual_seed(7)
        ts = [0, 1, 63, 64, 127, 128, 255, Ls - 1, Ls - 64, Ls - 129] + torch.randint(0, Ls, (sample,), generator=gen).tolist()
        rows = [(t, int(h)) for t, h in zip(ts, torch.randint(0, H, (len(ts),), generator=gen))]
    ref_o, ref_l = oracle.sys_prefill(q, k, v, rows)
    got_o = out.cpu().double().numpy()[[r[0] for r in rows], [r[1] for r in rows]]
    got_l = lse.cpu().double().numpy()[[r[0] for r in rows], [r[1] for r in rows]]
    T.check(got_o, ref_o, "prefill out")
    T.check(got_l, ref_l, "lse prefill")


# ----------------------------------------------------------------------------- rotary positions, decode loop
def _fp16_close(got, ref, what):
    """within fp16 rounding of the rotation (half an ulp, doubled) plus fp32 rounding of its unit-scale
    products (the rotation is computed in fp32)"""
    g = got.cpu().double().numpy()
    ok = ~np.isnan(ref)
    err = np.abs(g[ok] - ref[ok])
    assert np.all(err <= 2.0 ** -10 * np.abs(ref[ok]) + 2.0 ** -20), f"{what}: max err {err.max():.3e}"


@pytest.mark.parametrize("name,over", [("tiny_gqa", dict(Lq=3, chunk_requests=2)), ("llama2_7b", {}),
                                        ("llama2_13b_mixed", dict(Ls=32768))], ids=["gqa_chunks", "llama2_7b", "13b"])
def test_rope_positions(name, over):
    import shared_prompt_decode_gb300 as relay
    case = synth.make_case(synth.workload(name, **over), 51)
    g = T.to_dev(case)
    gk = torch.Generator().manual_seed(52)
    k_new = torch.randn(case.B, case.Lq, case.Hkv, case.D, generator=gk).half()
    q = g["q"].clone()
    kd = k_new.to(T.DEV)
    ws = relay.relay_rope(q, g["ctx_lens"], case.Ls, k_new=kd, q_lens=g["q_lens"])
    torch.cuda.synchronize()
    assert relay.device_status(ws) == 0
    _fp16_close(q, oracle.rope(case.q, case.Ls, case.ctx_lens, case.q_lens), "q")
    _fp16_close(kd, oracle.rope(k_new, case.Ls, case.ctx_lens, case.q_lens), "k_new")


# The attention layer's decode loop, several steps: rotate the step's new q
# and k at positions offset by the system prompt, append k and v to the pool,
# attend; the oracle runs the same loop on its own (its own rotation rounded
# to fp16, its own append) and every step's output is compared.
@pytest.mark.parametrize("name", ["llama2_7b", "tiny_gqa"])
def test_decode_loop(name):
    import shared_prompt_decode_gb300 as relay
    from dataclasses import replace
    steps = 4
    base_case = synth.make_case(name, 61)
    n0 = base_case.ctx_lens.clone()
    case = synth.make_case(name, 61, ctx_lens=[int(n) + steps for n in n0])   # tables with room for the new tokens
    g = T.to_dev(case)
    kc, vc = g["k_cache"].clone(), g["v_cache"].clone()
    ref_k, ref_v = case.k_cache.clone(), case.v_cache.clone()
    gen = torch.Generator().manual_seed(62)
    for step in range(steps):
        ctx = (n0 + step + 1).to(torch.int32)
        q = torch.randn(case.B, 1, case.H, case.D, generator=gen).half()
        k = torch.randn(case.B, 1, case.Hkv, case.D, generator=gen).half()
        v = torch.randn(case.B, 1, case.Hkv, case.D, generator=gen).half()
        # GPU: rotate, append, attend
        qd, kd, cd = q.to(T.DEV), k.to(T.DEV), ctx.to(T.DEV)
        relay.relay_rope(qd, cd, case.Ls, k_new=kd)
        relay.relay_kv_append(kd, v.to(T.DEV), g["block_tables"], cd, kc, vc)
        lse = torch.full((case.B, 1, case.H), float("nan"), dtype=torch.float32, device=T.DEV)
        out = relay.relay_attention_decode(qd, g["sys_k"], g["sys_v"], kc, vc, g["block_tables"], cd, lse_out=lse)
        torch.cuda.synchronize()
        # oracle: the same loop on its own
        qr = torch.from_numpy(oracle.rope(q, case.Ls, ctx).astype(np.float16))
        kr = torch.from_numpy(oracle.rope(k, case.Ls, ctx).astype(np.float16))
        cur = replace(case, q=qr, ctx_lens=ctx, k_cache=ref_k, v_cache=ref_v)
        ref_k, ref_v = oracle.kv_append(cur, kr, v)
        ref_o, ref_l = oracle.attention_full(replace(cur, k_cache=ref_k, v_cache=ref_v))
        T.check(out, ref_o, f"out (step {step})")
        T.check(lse, ref_l, f"lse (step {step})")


# ----------------------------------------------------------------------------- tree-shaped prefixes
# A global system prompt shared by every request and one group prompt per
# group of requests (a two-level prefix tree), then each request's context:
# relay_sys_attn over the global prompt (all rows) and over each group prompt
# (its group's rows, the others masked by q_lens = 0 and left at lse = -inf),
# relay_ctx_attn, and relay_fuse_n over the K = groups + 2 parts, against the
# oracle over each request's explicit concatenation [global; group; context].
def _tree_inputs(name, groups, Lp, seed):
    base = synth.make_case(name, seed)
    g = torch.Generator().manual_seed(seed + 1)
    grp = [((torch.randn(Lp, base.Hkv, base.D, generator=g) * base.wl.value_scale).half(),
            (torch.randn(Lp, base.Hkv, base.D, generator=g) * base.wl.value_scale).half()) for _ in range(groups)]
    return base, grp, [b % groups for b in range(base.B)]


def run_tree(base, grp, group_of, g=None):
    import shared_prompt_decode_gb300 as relay
    g = g or T.to_dev(base)
    o_parts, l_parts = [], []
    o, l = relay.relay_sys_attn(g["q"], g["sys_k"], g["sys_v"])
    o_parts.append(o)
    l_parts.append(l)
    for p, (k, v) in enumerate(grp):
        mask = torch.tensor([1 if group_of[b] == p else 0 for b in range(base.B)], dtype=torch.int32, device=T.DEV)
        o = torch.zeros(base.B, base.Lq, base.H, base.D, dtype=torch.float32, device=T.DEV)
        l = torch.full((base.B, base.Lq, base.H), float("-inf"), dtype=torch.float32, device=T.DEV)
        relay.relay_sys_attn(g["q"], k.to(T.DEV), v.to(T.DEV), q_lens=mask, o_sys=o, lse_sys=l)
        o_parts.append(o)
        l_parts.append(l)
    o, l = relay.relay_ctx_attn(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["ctx_lens"])
    o_parts.append(o)
    l_parts.append(l)
    lse = torch.full((base.B, base.Lq, base.H), float("nan"), dtype=torch.float32, device=T.DEV)
    out = relay.relay_fuse_n(o_parts, l_parts, lse_out=lse)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("name,groups,Lp", [("llama2_7b", 4, 512), ("tiny_gqa", 2, 40), ("tiny", 3, 0)],
                         ids=["llama2_7b_4groups", "gqa_2groups", "no_group_prompt"])
def test_tree_prefixes(name, groups, Lp):
    from dataclasses import replace
    base, grp, group_of = _tree_inputs(name, groups, Lp, 81)
    out, lse = run_tree(base, grp, group_of)
    got_o, got_l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    for p, (k, v) in enumerate(grp):
        flat = replace(base, sys_k=torch.cat([base.sys_k, k]), sys_v=torch.cat([base.sys_v, v]))
        ref_o, ref_l = oracle.attention_full(flat)
        idx = [b for b in range(base.B) if group_of[b] == p]
        T.check(got_o[idx], ref_o[idx], f"out (group {p})")
        T.check(got_l[idx], ref_l[idx], f"lse (group {p})")


# ----------------------------------------------------------------------------- shared prefix segments, one unit
# relay_attention_decode_prefixes: several shared segments (a global prompt
# and group prompts: a tree of shared prefixes), each request seeing the
# segments its mask selects, all fused in one streaming kernel and one merge;
# against the oracle over each request's explicit concatenation [its
# segments; its context].  Cases: the Llama-2-7B batch with a 2048-token
# global prompt and four 512-token group prompts; grouped-query heads; three
# segments with an empty one and requests that see none (pure context, or
# nothing at all); multi-row requests, on the streaming kernel and (64-row
# chunks at D = 128) with their contexts on the tensor cores.
PREFIX_CASES = [
    ("llama2_7b", {}, [2048, 512, 512, 512, 512], lambda b: 1 | (2 << (b % 4))),
    ("tiny_gqa", {}, [256, 40, 40], lambda b: 1 | (2 << (b % 2))),
    ("tiny", dict(pool_blocks=40), [100, 0, 77], lambda b: [0b101, 0b001, 0b000, 0b110][b]),
    ("tiny", dict(Lq=3, chunk_requests=2), [64, 130], lambda b: [1, 3, 2, 3][b]),
    # 64-row chunks at D = 128: their own contexts run on the tensor cores
    # while the segments stay on the streaming kernel
    ("llama2_7b", dict(B=6, Lq=64, chunk_requests=3), [300, 200], lambda b: [1, 3, 2, 3, 1, 2][b]),
]


@pytest.mark.parametrize("name,over,lens,mask_of", PREFIX_CASES,
                         ids=["llama2_7b_global_4groups", "gqa_2groups", "empty_and_unseen", "chunks",
                              "chunks_tensor_cores"])
def test_prefix_segments(name, over, lens, mask_of):
    import shared_prompt_decode_gb300 as relay
    from dataclasses import replace
    base = synth.make_case(synth.workload(name, **over), 91, ctx_lens=[0, 5, 0, 17] if name == "tiny" and
                           "pool_blocks" in over else None)
    gen = torch.Generator().manual_seed(92)
    segs = [((torch.randn(L, base.Hkv, base.D, generator=gen) * base.wl.value_scale).half(),
             (torch.randn(L, base.Hkv, base.D, generator=gen) * base.wl.value_scale).half()) for L in lens]
    masks = [mask_of(b) for b in range(base.B)]
    g = T.to_dev(base)
    lse = torch.full((base.B, base.Lq, base.H), float("nan"), dtype=torch.float32, device=T.DEV)
    out = torch.full_like(g["q"], float("nan"))
    relay.relay_attention_decode_prefixes(
        g["q"], [k.to(T.DEV) for k, _ in segs], [v.to(T.DEV) for _, v in segs],
        torch.tensor(masks, dtype=torch.int32, device=T.DEV), g["k_cache"], g["v_cache"], g["block_tables"],
        g["ctx_lens"], g["q_lens"], out=out, lse_out=lse, max_q_total=base.total_q() if base.q_lens is not None else 0)
    torch.cuda.synchronize()
    got_o, got_l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    for m in sorted(set(masks)):
        seen = [i for i in range(len(lens)) if (m >> i) & 1]
        k = torch.cat([segs[i][0] for i in seen]) if seen else torch.zeros(0, base.Hkv, base.D, dtype=torch.float16)
        v = torch.cat([segs[i][1] for i in seen]) if seen else torch.zeros(0, base.Hkv, base.D, dtype=torch.float16)
        flat = replace(base, sys_k=k, sys_v=v)
        ref_o, ref_l = oracle.attention_full(flat)
        idx = [b for b in range(base.B) if masks[b] == m]
        vm = T.valid_mask(base)[idx]
        T.check(got_o[idx][vm], ref_o[idx][vm], f"out (mask {m:b})")
        T.check(got_l[idx][vm], ref_l[idx][vm], f"lse (mask {m:b})")
    # rows past q_lens untouched
    ql = base.q_lens_list()
    for b in range(base.B):
        assert torch.isnan(out[b, ql[b]:].float()).all()
