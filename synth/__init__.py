"""Seeded synthetic inputs for relay decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CPU oracle and the CUDA path are fed from it,
so they see bit-identical fp16 inputs.

Workloads mirror the attention shapes of the RelayAttention study (arXiv
2402.14808: Llama-2-7B / 13B and Llama-30B heads, long shared system prompt,
batch 32 and up).  The pages measure end to end on ShareGPT/MMLU; those
datasets are not used: the synthetic shapes below stand in for them.

Layouts (all contiguous, row-major):
    q             [B, Lq, H, D]            fp16
    sys_k, sys_v  [Ls, Hkv, D]             fp16   shared system-prompt cache
    k_cache,
    v_cache       [num_blocks, Hkv, 16, D] fp16   paged context pool
                  (Hkv KV heads; Hkv = H unless the workload is grouped-query)
    block_tables  [B, max_blocks]          int32  unused entries are -1
    ctx_lens      [B]                      int32  context tokens per request
    q_lens        [B]                      int32  query rows per request
                                                  (None: every request has Lq)

Slots of the pool that hold no token (the tail of each request's last block
and the spare blocks) are filled with NaN, so any read that is not masked
shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

BLOCK_SIZE = 16


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    D: int
    Ls: int
    ctx_dist: tuple          # ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi) | ("fixed", n)
    value_scale: float       # q/k/v ~ N(0,1) * value_scale, stored fp16
    Lq: int = 1              # query-row stride of q / out
    chunk_requests: int = 0  # the last `chunk_requests` requests carry Lq query rows, the rest 1
    pool_blocks: Optional[int] = None   # fixed pool size (else needed blocks + 10% spare)
    spare_frac: float = 0.10
    Hkv: Optional[int] = None           # KV heads (None: H, multi-head)


# The five workloads.  Context-length draws are integer and inclusive.
WORKLOADS = {
    "tiny": Workload("tiny", B=4, H=4, D=64, Ls=256, ctx_dist=("uniform", 1, 64),
                     value_scale=1.0, pool_blocks=32),
    "llama2_7b": Workload("llama2_7b", B=32, H=32, D=128, Ls=2048,
                          ctx_dist=("uniform", 64, 1024), value_scale=0.5),
    "llama30b_sweep": Workload("llama30b_sweep", B=32, H=52, D=128, Ls=2048,
                               ctx_dist=("uniform", 128, 512), value_scale=0.5),
    "llama2_7b_b256": Workload("llama2_7b_b256", B=256, H=32, D=128, Ls=4096,
                               ctx_dist=("lognormal", 256.0, 1.0, 1, 2048), value_scale=0.5),
    "llama2_13b_mixed": Workload("llama2_13b_mixed", B=64, H=40, D=128, Ls=32768,
                                 ctx_dist=("uniform", 1, 4096), value_scale=0.5,
                                 Lq=128, chunk_requests=8),
    # Grouped-query attention (not on the pages; all five workloads above are
    # multi-head): the Llama-2-70B attention shape, 64 query heads over 8 KV
    # heads, with the Llama-2-7B workload's batch, prompt and contexts; and
    # small CPU-checkable grouped (2 KV heads) and multi-query (1) cases.
    "llama2_70b_gqa": Workload("llama2_70b_gqa", B=32, H=64, D=128, Ls=2048,
                               ctx_dist=("uniform", 64, 1024), value_scale=0.5, Hkv=8),
    "tiny_gqa": Workload("tiny_gqa", B=4, H=8, D=64, Ls=256, ctx_dist=("uniform", 1, 64),
                         value_scale=1.0, pool_blocks=32, Hkv=2),
    "tiny_mqa": Workload("tiny_mqa", B=4, H=4, D=64, Ls=256, ctx_dist=("uniform", 1, 64),
                         value_scale=1.0, pool_blocks=32, Hkv=1),
}

SWEEP_LS = (512, 1024, 2048, 4096, 8192, 16384)


def workload(name: str, **overrides) -> Workload:
    return replace(WORKLOADS[name], **overrides)


@dataclass
class Case:
    """One batch of inputs (torch CPU tensors)."""
    wl: Workload
    seed: int
    q: torch.Tensor
    sys_k: torch.Tensor
    sys_v: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    ctx_lens: torch.Tensor
    q_lens: Optional[torch.Tensor]
    extra: dict = field(default_factory=dict)

    @property
    def B(self): return self.q.shape[0]
    @property
    def Lq(self): return self.q.shape[1]
    @property
    def H(self): return self.q.shape[2]
    @property
    def D(self): return self.q.shape[3]
    @property
    def Ls(self): return self.sys_k.shape[0]
    @property
    def Hkv(self): return self.k_cache.shape[1]
    @property
    def num_blocks(self): return self.k_cache.shape[0]
    @property
    def max_blocks(self): return self.block_tables.shape[1]

    def q_lens_list(self):
        if self.q_lens is None:
            return [self.Lq] * self.B
        return [int(x) for x in self.q_lens]

    def total_q(self) -> int:
        return sum(self.q_lens_list())


def _draw_ctx_lens(wl: Workload, g: torch.Generator) -> list:
    kind = wl.ctx_dist[0]
    if kind == "uniform":
        lo, hi = wl.ctx_dist[1], wl.ctx_dist[2]
        lens = torch.randint(lo, hi + 1, (wl.B,), generator=g)
    elif kind == "lognormal":
        med, sigma, lo, hi = wl.ctx_dist[1:]
        z = torch.randn(wl.B, generator=g, dtype=torch.float64)
        lens = torch.clamp(torch.round(torch.exp(math.log(med) + sigma * z)), lo, hi).to(torch.int64)
    elif kind == "fixed":
        lens = torch.full((wl.B,), int(wl.ctx_dist[1]), dtype=torch.int64)
    else:
        raise ValueError(kind)
    return [int(x) for x in lens]


def _randn_f16(shape, g, scale):
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.float16)


def make_case(wl, seed: int = 0, ctx_lens: Optional[list] = None, q_lens: Optional[list] = None,
              poison: bool = True) -> Case:
    """Draw one seeded batch for workload `wl` (a Workload or its name).

    ctx_lens / q_lens override the drawn lengths (edge-case tests).  Chunk
    requests (the last `chunk_requests` indices) get Lq query rows and a
    context of at least Lq tokens; the query tokens are the last Lq positions
    of their context.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = torch.Generator().manual_seed(seed)
    B, H, D, Ls, Lq = wl.B, wl.H, wl.D, wl.Ls, wl.Lq
    Hkv = H if wl.Hkv is None else wl.Hkv
    assert H % Hkv == 0
    drawn = _draw_ctx_lens(wl, g)
    if ctx_lens is None:
        ctx_lens = drawn
    ctx_lens = [int(x) for x in ctx_lens]
    assert len(ctx_lens) == B
    if q_lens is None and wl.chunk_requests:
        q_lens = [1] * (B - wl.chunk_requests) + [Lq] * wl.chunk_requests
        ctx_lens = [max(n, Lq) if ql > 1 else n for n, ql in zip(ctx_lens, q_lens)]

    blocks_per_req = [-(-n // BLOCK_SIZE) for n in ctx_lens]
    max_blocks = max(1, max(blocks_per_req) if blocks_per_req else 1)
    needed = sum(blocks_per_req)
    if wl.pool_blocks is not None:
        num_blocks = max(wl.pool_blocks, needed)
    else:
        num_blocks = max(1, needed + int(math.ceil(wl.spare_frac * needed)))

    q = _randn_f16((B, Lq, H, D), g, wl.value_scale)
    sys_k = _randn_f16((Ls, Hkv, D), g, wl.value_scale)
    sys_v = _randn_f16((Ls, Hkv, D), g, wl.value_scale)
    k_cache = _randn_f16((num_blocks, Hkv, BLOCK_SIZE, D), g, wl.value_scale)
    v_cache = _randn_f16((num_blocks, Hkv, BLOCK_SIZE, D), g, wl.value_scale)

    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    block_tables = torch.full((B, max_blocks), -1, dtype=torch.int32)
    used = torch.zeros(num_blocks, BLOCK_SIZE, dtype=torch.bool)
    cursor = 0
    for b, nb in enumerate(blocks_per_req):
        ids = perm[cursor:cursor + nb]
        cursor += nb
        block_tables[b, :nb] = ids
        for j in range(nb):
            valid = min(BLOCK_SIZE, ctx_lens[b] - j * BLOCK_SIZE)
            used[int(ids[j]), :valid] = True
    if poison:
        nan = torch.tensor(float("nan"), dtype=torch.float16)
        mask = (~used)[:, None, :, None].expand_as(k_cache)
        k_cache[mask] = nan
        v_cache[mask] = nan

    ql = None if q_lens is None else torch.tensor(q_lens, dtype=torch.int32)
    if ql is not None:
        assert all(0 <= x <= Lq for x in q_lens)
        # Rows beyond a request's query length are padding: poison them too.
        if poison:
            for b, n in enumerate(q_lens):
                q[b, n:] = float("nan")
    return Case(wl, seed, q, sys_k, sys_v, k_cache, v_cache, block_tables,
                torch.tensor(ctx_lens, dtype=torch.int32), ql)


def relabel_pool(case: Case, seed: int) -> Case:
    """Same logical inputs with the pool's physical blocks permuted and the
    tables rewritten to match (a pure relabelling: no value changes)."""
    g = torch.Generator().manual_seed(seed)
    nb = case.num_blocks
    new_of_old = torch.randperm(nb, generator=g)
    k = torch.empty_like(case.k_cache)
    v = torch.empty_like(case.v_cache)
    k[new_of_old] = case.k_cache
    v[new_of_old] = case.v_cache
    bt = case.block_tables.clone()
    valid = bt >= 0
    bt[valid] = new_of_old[bt[valid].long()].to(torch.int32)
    return replace(case, k_cache=k, v_cache=v, block_tables=bt)


def with_system_in_pool(case: Case):
    """Copy the system-prompt cache into extra blocks appended to the pool.

    Returns (k_pool, v_pool, sys_block_ids): the layout a prefix-sharing
    paged-attention system uses, where every request's table begins with the
    shared system blocks.  The tail of the last system block is NaN.
    """
    Ls, H, D = case.Ls, case.Hkv, case.D
    n_sys = -(-Ls // BLOCK_SIZE)
    pad = n_sys * BLOCK_SIZE - Ls
    def to_blocks(x):
        if pad:
            x = torch.cat([x, torch.full((pad, H, D), float("nan"), dtype=x.dtype)], 0)
        return x.reshape(n_sys, BLOCK_SIZE, H, D).permute(0, 2, 1, 3).contiguous()
    k_pool = torch.cat([case.k_cache, to_blocks(case.sys_k)], 0)
    v_pool = torch.cat([case.v_cache, to_blocks(case.sys_v)], 0)
    ids = torch.arange(case.num_blocks, case.num_blocks + n_sys, dtype=torch.int32)
    return k_pool, v_pool, ids


def sample_rows(case: Case, n: int, seed: int):
    """A seeded sample of (b, i, h) output rows, i < q_lens[b]."""
    g = torch.Generator().manual_seed(seed)
    ql = case.q_lens_list()
    pairs = [(b, i) for b in range(case.B) for i in range(ql[b])]
    if not pairs:
        return []
    idx = torch.randint(0, len(pairs), (n,), generator=g)
    hs = torch.randint(0, case.H, (n,), generator=g)
    return [(pairs[int(k)][0], pairs[int(k)][1], int(h)) for k, h in zip(idx, hs)]
