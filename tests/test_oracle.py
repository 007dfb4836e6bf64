"""Pins for the CPU oracle (no GPU).

The pages print no output values, so the oracle is pinned by what the
mathematics fixes: a hand-worked example, closed forms, brute force with
explicit numpy matrices, torch's fp64 scaled-dot-product attention over the
explicit concatenation, the relay identity (the three steps reproduce the
direct definition), the empty-segment special cases, and invariance under
relabelling of the paged pool.  Each check is chosen so that a plausible
slip in the oracle (a wrong causal offset, a swapped head/token index, a
dropped scale, a wrong fusion weight, a mis-decoded fp16) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


# ----------------------------------------------------------------------------- helpers
def _resolve(x):
    if isinstance(x, list):
        if x and isinstance(x[0], str):
            if x[0] == "frac":
                return x[1] / x[2]
            if x[0] == "ln":
                return math.log(x[1])
            raise ValueError(x)
        return [_resolve(y) for y in x]
    return float(x)


def _flat(x):
    r = _resolve(x)
    return np.array(r, dtype=np.float64).ravel()


def _case_from_golden(ex):
    B, Lq, H, D = ex["B"], ex["Lq"], ex["H"], ex["D"]
    q = torch.tensor(ex["q"], dtype=torch.float16).reshape(B, Lq, H, D)
    sk = torch.tensor(ex["sys_k"], dtype=torch.float16).reshape(-1, H, D)
    sv = torch.tensor(ex["sys_v"], dtype=torch.float16).reshape(-1, H, D)
    nb = ex["pool_blocks"]
    kc = torch.full((nb, H, 16, D), float("nan"), dtype=torch.float16)
    vc = torch.full((nb, H, 16, D), float("nan"), dtype=torch.float16)
    bt = torch.tensor(ex["block_table"], dtype=torch.int32)
    ck = torch.tensor(ex["ctx_tokens_k"], dtype=torch.float16).reshape(-1, H, D)
    cv = torch.tensor(ex["ctx_tokens_v"], dtype=torch.float16).reshape(-1, H, D)
    for t in range(ck.shape[0]):     # single request in the examples
        blk = int(bt[0, t // 16])
        kc[blk, :, t % 16] = ck[t]
        vc[blk, :, t % 16] = cv[t]
    ql = None if ex["q_lens"] is None else torch.tensor(ex["q_lens"], dtype=torch.int32)
    wl = synth.Workload("golden", B=B, H=H, D=D, Ls=sk.shape[0], ctx_dist=("fixed", 0),
                        value_scale=1.0, Lq=Lq)
    return synth.Case(wl, 0, q, sk, sv, kc, vc, bt, torch.tensor(ex["ctx_lens"], dtype=torch.int32), ql)


def _small_case(seed, B=2, H=2, D=8, Ls=5, Lq=1, ctx=None, q_lens=None, scale=1.0):
    wl = synth.Workload("small", B=B, H=H, D=D, Ls=Ls, ctx_dist=("uniform", 0, 8),
                        value_scale=scale, Lq=Lq, pool_blocks=4)
    return synth.make_case(wl, seed, ctx_lens=ctx, q_lens=q_lens)


def _numpy_brute(case, scale):
    """Independent restatement with explicit matrices: for each (b, h) build
    the full key matrix [system; context] and a boolean visibility matrix from
    absolute positions, then a row softmax."""
    q = case.q.double().numpy()
    sk = case.sys_k.double().numpy()
    sv = case.sys_v.double().numpy()
    kc = case.k_cache.double().numpy()
    vc = case.v_cache.double().numpy()
    bt = case.block_tables.numpy()
    ql = case.q_lens_list()
    out = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:3], np.nan)
    for b in range(case.B):
        n = int(case.ctx_lens[b])
        for h in range(case.H):
            ctxk = np.stack([kc[bt[b, t // 16], h, t % 16] for t in range(n)]) if n else np.zeros((0, case.D))
            ctxv = np.stack([vc[bt[b, t // 16], h, t % 16] for t in range(n)]) if n else np.zeros((0, case.D))
            K = np.concatenate([sk[:, h], ctxk], 0)
            V = np.concatenate([sv[:, h], ctxv], 0)
            key_pos = np.arange(K.shape[0])
            for i in range(ql[b]):
                # system keys precede every request token; context key t is
                # visible to the row whose token sits at context position n-ql+i
                vis = (key_pos < case.Ls) | (key_pos - case.Ls <= n - ql[b] + i)
                if not vis.any():
                    out[b, i, h] = 0.0
                    lse[b, i, h] = -np.inf
                    continue
                s = scale * (K[vis] @ q[b, i, h])
                m = s.max()
                e = np.exp(s - m)
                out[b, i, h] = (e / e.sum()) @ V[vis]
                lse[b, i, h] = m + np.log(e.sum())
    return out, lse


# ----------------------------------------------------------------------------- pins
def test_half_decoder_matches_numpy(oracle_lib):
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle_lib.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.parametrize("idx", [0, 1])
def test_golden_hand_examples(oracle_lib, idx):
    ex = json.load(open(GOLDEN))["examples"][idx]
    case = _case_from_golden(ex)
    sc = math.log(2.0)
    for part, exp in ex["expect"].items():
        if part == "alpha_sys":
            continue
        out, lse = oracle_lib.attention_full(case, part, scale=sc)
        np.testing.assert_allclose(out.ravel(), _flat(exp["out"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse.ravel(), _flat(exp["lse"]), rtol=0, atol=1e-12)
    if "alpha_sys" in ex["expect"]:
        os_, ls = oracle_lib.attention_full(case, "sys", scale=sc)
        oc, lc = oracle_lib.attention_full(case, "ctx", scale=sc)
        of, lf, a = oracle_lib.relay_fuse(os_, ls, oc, lc)
        np.testing.assert_allclose(a.ravel(), _flat(ex["expect"]["alpha_sys"]), atol=1e-12)
        np.testing.assert_allclose(of.ravel(), _flat(ex["expect"]["full"]["out"]), atol=1e-12)


def test_single_key_returns_its_value(oracle_lib):
    case = _small_case(1, B=1, H=2, D=8, Ls=1, ctx=[0])
    out, lse = oracle_lib.attention_full(case)
    v = case.sys_v.double().numpy()[0]
    np.testing.assert_array_equal(out[0, 0], v)
    s = (case.q.double().numpy()[0, 0] * case.sys_k.double().numpy()[0]).sum(-1) / math.sqrt(8)
    np.testing.assert_allclose(lse[0, 0], s, atol=1e-12)


def test_equal_scores_give_mean_of_values(oracle_lib):
    case = _small_case(2, B=2, H=2, D=8, Ls=5, ctx=[7, 3])
    case.sys_k.zero_()
    case.k_cache.zero_()
    out, lse = oracle_lib.attention_full(case)
    for b in range(2):
        n = int(case.ctx_lens[b])
        for h in range(2):
            vals = [case.sys_v[t, h].double() for t in range(5)]
            vals += [case.v_cache[int(case.block_tables[b, t // 16]), h, t % 16].double() for t in range(n)]
            np.testing.assert_allclose(out[b, 0, h], torch.stack(vals).mean(0).numpy(), atol=1e-12)
            np.testing.assert_allclose(lse[b, 0, h], math.log(5 + n), atol=1e-12)


@pytest.mark.parametrize("seed,Lq,q_lens,ctx,Ls", [
    (3, 1, None, [5, 8], 5),
    (4, 3, [3, 1], [8, 2], 4),
    (5, 3, [2, 3], [1, 6], 0),    # more query rows than context for b=0 (visibility clips at 0)
    (6, 2, [2, 2], [0, 7], 3),
])
def test_brute_force_numpy(oracle_lib, seed, Lq, q_lens, ctx, Ls):
    case = _small_case(seed, B=2, H=2, D=8, Ls=Ls, Lq=Lq, ctx=ctx, q_lens=q_lens)
    sc = 1.0 / math.sqrt(8)
    o_ref, l_ref = _numpy_brute(case, sc)
    o, l = oracle_lib.attention_full(case)
    ok = ~np.isnan(l_ref)
    np.testing.assert_allclose(o[ok], o_ref[ok], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l[ok], l_ref[ok], rtol=0, atol=1e-13)


@pytest.mark.parametrize("q_lens", [None, [1, 3, 2, 3]])
def test_sdpa_fp64_over_concatenation(oracle_lib, q_lens):
    wl = synth.workload("tiny", Lq=1 if q_lens is None else 3)
    case = synth.make_case(wl, seed=7, q_lens=q_lens)
    o, l = oracle_lib.attention_full(case)
    q = case.q.double()
    for b in range(case.B):
        n = int(case.ctx_lens[b])
        t = torch.arange(n)
        blk = case.block_tables[b, (t // 16)].long()
        kc = case.k_cache[blk, :, t % 16].double()       # [n, H, D]
        vc = case.v_cache[blk, :, t % 16].double()
        K = torch.cat([case.sys_k.double(), kc], 0).transpose(0, 1)   # [H, L, D]
        V = torch.cat([case.sys_v.double(), vc], 0).transpose(0, 1)
        ql = case.q_lens_list()[b]
        qpos = n - ql + torch.arange(ql)                                    # context position of each query token
        kpos = torch.arange(K.shape[1]) - case.Ls
        mask = (kpos[None, :] < 0) | (kpos[None, :] <= qpos[:, None])     # [ql, L]
        Q = q[b, :ql].transpose(0, 1)                                       # [H, ql, D]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
        np.testing.assert_allclose(o[b, :ql], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def _relay_decomposed(oracle_lib, case):
    rows = oracle_lib.all_rows(case)
    os_, ls = oracle_lib.attention_rows(case, rows, "sys")
    oc, lc = oracle_lib.attention_rows(case, rows, "ctx")
    of, lf, a = oracle_lib.relay_fuse(os_, ls, oc, lc)
    od, ld = oracle_lib.attention_rows(case, rows, "full")
    return rows, (os_, ls, oc, lc, of, lf, a), (od, ld)


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("llama30b_sweep", dict(B=3, H=3, Ls=512)),
    ("llama2_7b_b256", dict(B=5, H=2, Ls=128)),
    ("llama2_13b_mixed", dict(B=6, H=2, Ls=256, Lq=8, chunk_requests=2, ctx_dist=("uniform", 1, 96))),
    ("tiny_gqa", {}),
    ("tiny_mqa", dict(Lq=3, chunk_requests=2)),
])
def test_relay_identity(oracle_lib, name, over):
    case = synth.make_case(synth.workload(name, **over), seed=11)
    rows, (os_, ls, oc, lc, of, lf, a), (od, ld) = _relay_decomposed(oracle_lib, case)
    np.testing.assert_allclose(of, od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lf, ld, rtol=0, atol=1e-12)
    # fusion weights: convex, and equal to the system part's share of the softmax mass
    ne = ~np.isnan(a)
    assert np.all((a[ne] >= 0) & (a[ne] <= 1))
    np.testing.assert_allclose(a[ne], np.exp(ls[ne] - ld[ne]), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose((1 - a[ne]), np.exp(lc[ne] - ld[ne]), rtol=1e-9, atol=1e-15)
    assert np.all(np.isfinite(od))


def test_empty_context_is_system_attention(oracle_lib):
    case = synth.make_case("tiny", seed=3, ctx_lens=[0, 5, 0, 17])
    o, l = oracle_lib.attention_full(case)
    os_, ls = oracle_lib.attention_full(case, "sys")
    oc, lc = oracle_lib.attention_full(case, "ctx")
    for b in (0, 2):
        np.testing.assert_array_equal(o[b], os_[b])
        np.testing.assert_array_equal(l[b], ls[b])
        assert np.all(lc[b] == -np.inf) and np.all(oc[b] == 0)


def test_empty_system_is_context_attention(oracle_lib):
    case = synth.make_case(synth.workload("tiny", Ls=0), seed=3)
    o, l = oracle_lib.attention_full(case)
    oc, lc = oracle_lib.attention_full(case, "ctx")
    np.testing.assert_array_equal(o, oc)
    np.testing.assert_array_equal(l, lc)


def test_both_empty_gives_zero_and_neg_inf(oracle_lib):
    case = synth.make_case(synth.workload("tiny", Ls=0), seed=3, ctx_lens=[0, 0, 4, 0])
    o, l = oracle_lib.attention_full(case)
    for b in (0, 1, 3):
        assert np.all(o[b] == 0) and np.all(l[b] == -np.inf)
    _, _, a = oracle_lib.relay_fuse(*oracle_lib.attention_full(case, "sys"), *oracle_lib.attention_full(case, "ctx"))
    assert np.all(np.isnan(a[[0, 1, 3]]))


def test_pool_relabelling_is_invisible(oracle_lib):
    case = synth.make_case("tiny", seed=5)
    o1, l1 = oracle_lib.attention_full(case)
    c2 = synth.relabel_pool(case, seed=9)
    assert not torch.equal(c2.block_tables, case.block_tables)
    o2, l2 = oracle_lib.attention_full(c2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_poisoned_slots_never_read(oracle_lib):
    case = synth.make_case("tiny", seed=6)
    assert torch.isnan(case.k_cache).any()
    o, l = oracle_lib.attention_full(case)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))


def test_bad_block_id_rejected(oracle_lib):
    case = synth.make_case("tiny", seed=6)
    case.block_tables[1, 0] = case.num_blocks
    with pytest.raises(ValueError):
        oracle_lib.attention_rows(case, [(1, 0, 0)])


def test_scale_is_applied(oracle_lib):
    case = _small_case(8, B=1, H=1, D=8, Ls=4, ctx=[3])
    o1, l1 = oracle_lib.attention_full(case, scale=0.5)
    o2, l2 = oracle_lib.attention_full(case, scale=1.0)
    assert not np.allclose(o1, o2)
    o_ref, l_ref = _numpy_brute(case, 0.5)
    np.testing.assert_allclose(o1, o_ref, atol=1e-13)


# ----------------------------------------------------------------------------- grouped-query heads
# Query head h reads KV head h / (H / Hkv).  Two pins that do not restate that
# formula: the multi-head oracle (pinned above) over caches whose KV heads are
# expanded with torch.repeat_interleave, and torch's fp64 scaled-dot-product
# attention with its own grouped-query option.  Both fail for a wrong
# grouping (for example h % Hkv).
def _expand_kv(case):
    G = case.H // case.Hkv
    ex = lambda t: t.repeat_interleave(G, dim=1).contiguous()
    from dataclasses import replace
    return synth.Case(replace(case.wl, Hkv=None), case.seed, case.q, ex(case.sys_k), ex(case.sys_v),
                      ex(case.k_cache), ex(case.v_cache), case.block_tables, case.ctx_lens, case.q_lens)


@pytest.mark.parametrize("name,over", [
    ("tiny_gqa", {}),
    ("tiny_mqa", {}),
    ("tiny_gqa", dict(Lq=3, chunk_requests=2)),
    ("tiny_gqa", dict(H=8, Hkv=4, Ls=0)),
])
def test_gqa_equals_multi_head_on_expanded_kv(oracle_lib, name, over):
    case = synth.make_case(synth.workload(name, **over), seed=13)
    assert case.Hkv < case.H
    full = _expand_kv(case)
    assert full.Hkv == full.H
    o, l = oracle_lib.attention_full(case)
    o2, l2 = oracle_lib.attention_full(full)
    ok = ~np.isnan(l2)
    np.testing.assert_array_equal(o[ok], o2[ok])
    np.testing.assert_array_equal(l[ok], l2[ok])


@pytest.mark.parametrize("name", ["tiny_gqa", "tiny_mqa"])
def test_gqa_sdpa_fp64(oracle_lib, name):
    case = synth.make_case(name, seed=17)
    o, l = oracle_lib.attention_full(case)
    q = case.q.double()
    for b in range(case.B):
        n = int(case.ctx_lens[b])
        t = torch.arange(n)
        blk = case.block_tables[b, (t // 16)].long()
        kc = case.k_cache[blk, :, t % 16].double()                            # [n, Hkv, D]
        vc = case.v_cache[blk, :, t % 16].double()
        K = torch.cat([case.sys_k.double(), kc], 0).transpose(0, 1)         # [Hkv, L, D]
        V = torch.cat([case.sys_v.double(), vc], 0).transpose(0, 1)
        Q = q[b, :1].transpose(0, 1)                                         # [H, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, enable_gqa=True)
        np.testing.assert_allclose(o[b, :1], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- KV append
# Append then attend must equal attention over the explicit concatenation
# [system; the context before the new tokens, read from the original pool;
# the new rows] with the causal mask: a row written to the wrong slot, head
# or request changes the result.
@pytest.mark.parametrize("name,over", [("tiny", dict(Lq=3, chunk_requests=2)), ("tiny_gqa", dict(Lq=2, chunk_requests=4))])
def test_kv_append_then_attend_equals_concatenation(oracle_lib, name, over):
    from dataclasses import replace
    case = synth.make_case(synth.workload(name, **over), seed=29)
    g = torch.Generator().manual_seed(5)
    shape = (case.B, case.Lq, case.Hkv, case.D)
    k_new = torch.randn(*shape, generator=g).half()
    v_new = torch.randn(*shape, generator=g).half()
    kc2, vc2 = oracle_lib.kv_append(case, k_new, v_new)
    o, l = oracle_lib.attention_full(replace(case, k_cache=kc2, v_cache=vc2))
    q = case.q.double()
    for b in range(case.B):
        n, ql = int(case.ctx_lens[b]), case.q_lens_list()[b]
        old = n - ql
        t = torch.arange(old)
        blk = case.block_tables[b, t // 16].long()
        K = torch.cat([case.sys_k.double(), case.k_cache[blk, :, t % 16].double(), k_new[b, :ql].double()], 0)
        V = torch.cat([case.sys_v.double(), case.v_cache[blk, :, t % 16].double(), v_new[b, :ql].double()], 0)
        kpos = torch.arange(K.shape[0]) - case.Ls                   # context position of each key (< 0: system)
        mask = (kpos[None, :] < 0) | (kpos[None, :] <= old + torch.arange(ql)[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(q[b, :ql].transpose(0, 1), K.transpose(0, 1),
                                                               V.transpose(0, 1), attn_mask=mask, enable_gqa=True)
        np.testing.assert_allclose(o[b, :ql], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_kv_append_rejects_bad_input(oracle_lib):
    case = synth.make_case(synth.workload("tiny", Lq=2, chunk_requests=2), seed=31)
    k_new = torch.zeros(case.B, case.Lq, case.Hkv, case.D, dtype=torch.float16)
    bad = case.block_tables.clone()
    bad[bad >= 0] = case.num_blocks                                 # every used block id out of range
    from dataclasses import replace
    with pytest.raises(ValueError):
        oracle_lib.kv_append(replace(case, block_tables=bad), k_new, k_new)
    short = case.ctx_lens.clone()
    short[-1] = 1                                                   # a 2-row request with a 1-token context
    with pytest.raises(ValueError):
        oracle_lib.kv_append(replace(case, ctx_lens=short), k_new, k_new)


# ----------------------------------------------------------------------------- system-prompt prefill
# Causal self-attention of the system prompt: torch's fp64 scaled-dot-product
# attention with its own causal and grouped-query options, and row t against
# the (pinned) decode oracle attending one query over the first t+1 system
# tokens with no context.
def _prefill_inputs(Ls, H, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Ls, H, D, generator=g).half()
    k = torch.randn(Ls, Hkv, D, generator=g).half()
    v = torch.randn(Ls, Hkv, D, generator=g).half()
    return q, k, v


@pytest.mark.parametrize("Ls,H,Hkv", [(40, 4, 4), (37, 4, 2), (20, 3, 1)])
def test_sys_prefill_sdpa_causal(oracle_lib, Ls, H, Hkv):
    D = 16
    q, k, v = _prefill_inputs(Ls, H, Hkv, D, 3)
    o, l = oracle_lib.sys_prefill(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double().transpose(0, 1), k.double().transpose(0, 1),
                                                           v.double().transpose(0, 1), is_causal=True,
                                                           enable_gqa=True)
    np.testing.assert_allclose(o.reshape(Ls, H, D), ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_sys_prefill_row_is_decode_over_prefix(oracle_lib):
    Ls, H, Hkv, D = 24, 4, 2, 8
    q, k, v = _prefill_inputs(Ls, H, Hkv, D, 4)
    rows = [(t, h) for t in (0, 1, 7, 23) for h in range(H)]
    o, l = oracle_lib.sys_prefill(q, k, v, rows)
    for n, (t, h) in enumerate(rows):
        wl = synth.Workload("prefix", B=1, H=H, D=D, Ls=t + 1, ctx_dist=("fixed", 0), value_scale=1.0, Hkv=Hkv)
        case = synth.Case(wl, 0, q[t][None, None].contiguous(), k[:t + 1].contiguous(), v[:t + 1].contiguous(),
                          torch.zeros(1, Hkv, 16, D, dtype=torch.float16), torch.zeros(1, Hkv, 16, D, dtype=torch.float16),
                          torch.zeros(1, 1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32), None)
        od, ld = oracle_lib.attention_rows(case, [(0, 0, h)], "sys")
        np.testing.assert_allclose(o[n], od[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(l[n], ld[0], rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- rotary positions
# Rows sit at position Ls + ctx_len - q_len + i.  Pins from the mathematics
# of the rotation: a D = 2 head turns by exactly the position; in a D = 4 head
# pair 1 turns by p / sqrt(base); position 0 is the identity; rotations keep
# pair norms; and scores depend only on relative positions.
def _rope1(oracle_lib, vec, Ls, n, base=10000.0):
    x = torch.tensor(vec, dtype=torch.float16).reshape(1, 1, 1, -1)
    return oracle_lib.rope(x, Ls, torch.tensor([n], dtype=torch.int32), None, base)[0, 0, 0]


def test_rope_closed_forms(oracle_lib):
    for Ls, n in [(0, 1), (5, 3), (1000, 1), (32768, 4096)]:
        p = Ls + n - 1
        o = _rope1(oracle_lib, [1.0, 0.0], Ls, n)
        np.testing.assert_allclose(o, [math.cos(p), math.sin(p)], rtol=0, atol=1e-12)
        o = _rope1(oracle_lib, [0.0, 1.0, 0.0, 0.0], Ls, n, base=400.0)
        ang = p / 20.0                                            # p * 400^(-2/4)
        np.testing.assert_allclose(o, [0.0, math.cos(ang), 0.0, math.sin(ang)], rtol=0, atol=1e-12)


def test_rope_identity_norms_and_relative_positions(oracle_lib):
    g = torch.Generator().manual_seed(8)
    x = torch.randn(2, 1, 3, 16, generator=g).half()
    y = torch.randn(2, 1, 3, 16, generator=g).half()
    one = torch.ones(2, dtype=torch.int32)
    np.testing.assert_array_equal(oracle_lib.rope(x, 0, one), x.double().numpy())     # position 0
    ctx = torch.tensor([7, 300], dtype=torch.int32)
    rx = oracle_lib.rope(x, 11, ctx)
    pairs = lambda a: np.hypot(a[..., :8], a[..., 8:])
    np.testing.assert_allclose(pairs(rx), pairs(x.double().numpy()), rtol=1e-13)
    for shift in (1, 1000):
        a = (oracle_lib.rope(x, 11, ctx) * oracle_lib.rope(y, 4, ctx)).sum(-1)
        b = (oracle_lib.rope(x, 11 + shift, ctx) * oracle_lib.rope(y, 4 + shift, ctx)).sum(-1)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)


# ----------------------------------------------------------------------------- tree-shaped prefixes
# A two-level tree: a global prompt shared by every request, a group prompt
# shared by some, then each request's context.  Attention over the explicit
# concatenation [global; group; context] equals the cascaded relay fusion
# fuse(fuse(global, group), context), built from the oracle's (pinned)
# two-part fusion: the LSE merge is associative.
def test_cascaded_fusion_equals_concatenation(oracle_lib):
    from dataclasses import replace
    base = synth.make_case(synth.workload("tiny_gqa", Ls=48), seed=71)
    g = torch.Generator().manual_seed(72)
    grp_k = torch.randn(20, base.Hkv, base.D, generator=g).half()
    grp_v = torch.randn(20, base.Hkv, base.D, generator=g).half()
    flat = replace(base, sys_k=torch.cat([base.sys_k, grp_k]), sys_v=torch.cat([base.sys_v, grp_v]))
    od, ld = oracle_lib.attention_full(flat)
    rows = oracle_lib.all_rows(base)
    og, lg = oracle_lib.attention_rows(base, rows, "sys")
    op, lp = oracle_lib.attention_rows(replace(base, sys_k=grp_k, sys_v=grp_v), rows, "sys")
    oc, lc = oracle_lib.attention_rows(base, rows, "ctx")
    o1, l1, _ = oracle_lib.relay_fuse(og, lg, op, lp)
    o2, l2, _ = oracle_lib.relay_fuse(o1, l1, oc, lc)
    for n, (b, i, h) in enumerate(rows):
        np.testing.assert_allclose(o2[n], od[b, i, h], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2[n], ld[b, i, h], rtol=0, atol=1e-12)
