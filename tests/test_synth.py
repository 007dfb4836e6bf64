"""The seeded input generator: shapes, distributions, pool structure (no GPU)."""
import torch

import synth


def test_llama2_7b_shapes_and_ranges():
    c = synth.make_case("llama2_7b", seed=0)
    assert c.q.shape == (32, 1, 32, 128) and c.q.dtype == torch.float16
    assert c.sys_k.shape == (2048, 32, 128)
    assert c.k_cache.shape[1:] == (32, 16, 128)
    assert int(c.ctx_lens.min()) >= 64 and int(c.ctx_lens.max()) <= 1024
    # pool = needed blocks + 10% spare, every used id distinct
    used = c.block_tables[c.block_tables >= 0]
    assert used.numel() == sum(-(-int(n) // 16) for n in c.ctx_lens)
    assert used.unique().numel() == used.numel()
    assert c.num_blocks == used.numel() + -(-used.numel() // 10)


def test_seed_determinism():
    a = synth.make_case("tiny", seed=3)
    b = synth.make_case("tiny", seed=3)
    assert torch.equal(a.q, b.q) and torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.k_cache.nan_to_num(), b.k_cache.nan_to_num())


def test_unused_slots_are_nan_and_used_slots_finite():
    c = synth.make_case("tiny", seed=1)
    for b in range(c.B):
        n = int(c.ctx_lens[b])
        for t in range(-(-n // 16) * 16):
            blk = int(c.block_tables[b, t // 16])
            slot = c.k_cache[blk, :, t % 16]
            assert torch.isfinite(slot).all() == (t < n)


def test_lognormal_and_mixed():
    c = synth.make_case("llama2_7b_b256", seed=0)
    assert int(c.ctx_lens.min()) >= 1 and int(c.ctx_lens.max()) <= 2048
    m = synth.make_case(synth.workload("llama2_13b_mixed", B=16, H=2, Ls=64), seed=0)
    ql = m.q_lens_list()
    assert ql[:8] == [1] * 8 and ql[8:] == [128] * 8
    assert all(int(m.ctx_lens[b]) >= 128 for b in range(8, 16))
    assert torch.isnan(m.q[0, 1:]).all()


def test_relabel_and_system_pool():
    c = synth.make_case("tiny", seed=2)
    r = synth.relabel_pool(c, 4)
    for b in range(c.B):
        for j in range(-(-int(c.ctx_lens[b]) // 16)):
            assert torch.equal(c.k_cache[int(c.block_tables[b, j])].nan_to_num(7.0),
                               r.k_cache[int(r.block_tables[b, j])].nan_to_num(7.0))
    kp, vp, ids = synth.with_system_in_pool(c)
    assert ids.numel() == 16
    assert torch.equal(kp[int(ids[1]), :, 3], c.sys_k[19])
