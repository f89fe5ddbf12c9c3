"""Seeded synthetic workspaces for per-step working-set recall.

This module only draws random numbers and arranges them in the library's
layouts; it holds none of the recall arithmetic (no RoPE, no Mean-K, no
scoring), so both the CUDA path and the CPU oracle can consume its output.

Recipe (all draws from one ``torch.Generator`` seeded with ``seed``, in the
order listed):

1. ``u``: one random unit direction of length ``head_dim`` (normalised N(0,1)).
   The churn workload draws ``n_topics`` such directions instead.
2. Planted blocks: ``n_planted`` (or ``round(planted_frac * N)``) block ids drawn
   without replacement from the non-reserved range ``[S, N - W)``.
3. Raw (position-independent) K and V of the history, i.i.d. N(0, k_std^2), in
   page layout ``[block][layer][kv_head][32][head_dim]``.  The raw K of every
   token of a planted block is shifted by ``k_shift * k_std * u`` in every layer
   and KV head, so its Mean-K carries the shift.
4. RoPE-free queries ``[layer][query][q_head][head_dim]`` drawn N(0,1) and shifted
   by ``q_shift * u`` (churn: query ``m`` of step ``t`` is shifted along the
   topic ``A_t[m mod topics_per_step]``).

Values are drawn in fp32 and rounded once to the storage dtype (bf16 RNE via
``Tensor.to``; e4m3 through torch's float8_e4m3fn, kept as uint8 bit patterns).  The workspaces of KVMem (Virtualizing Million-Token Agent
Workspaces on a Consumer GPU, §6) are real agent traces that are not available
here; these draws stand in for them with the same shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from .configs import BLOCK_TOKENS, Workload

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


def _to_storage(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """float32 values as the storage dtype (uint8 holds e4m3 bit patterns)."""
    if dtype == torch.uint8:
        return x.to(torch.float8_e4m3fn).view(torch.uint8)
    return x.to(dtype)


def _from_storage(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.uint8:
        return x.view(torch.float8_e4m3fn).float()
    return x.float()


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device, chunk_elems=1 << 28, out_dtype=torch.float32, scale=1.0):
    """N(0, scale^2) in ``out_dtype``, drawn in fp32 chunks to bound peak memory."""
    out = torch.empty(shape, dtype=out_dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        tmp = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            tmp.mul_(scale)
        flat[s:e].copy_(_to_storage(tmp, out_dtype))
    return out


def unit_vectors(n: int, d: int, gen, device) -> torch.Tensor:
    u = torch.randn(n, d, generator=gen, device=device, dtype=torch.float32)
    return u / u.norm(dim=1, keepdim=True)


def planted_blocks(wl: Workload, n_blocks: int, gen) -> torch.Tensor:
    # candidates lie between the sink and the recent blocks; a history shorter
    # than the reserved blocks has none
    lo, hi = wl.sink_blocks, n_blocks - wl.recent_blocks
    span = max(0, hi - lo)
    n = wl.n_planted if wl.n_planted > 0 else int(round(wl.planted_frac * n_blocks))
    n = max(0, min(n, span))
    perm = torch.randperm(span, generator=gen, device=gen.device)[:n] + lo
    return torch.sort(perm).values.to(torch.int64)


@dataclass
class Workspace:
    wl: Workload
    u: torch.Tensor                      # [d] or [n_topics, d] fp32
    planted: torch.Tensor                # int64 block ids
    raw_k: torch.Tensor | None = None    # [N][L][G][32][d]
    v: torch.Tensor | None = None        # [N][L][G][32][d]
    q: torch.Tensor | None = None        # [L][M_q][H][d]
    index: torch.Tensor | None = None    # [L][G][N][d] (drawn directly)
    topic_of: torch.Tensor | None = None  # planted block -> topic (churn)
    extra: dict = field(default_factory=dict)


def make_workspace(wl: Workload, seed: int = 0, device="cpu", n_blocks: int | None = None,
                   with_kv: bool = True, with_q: bool = True) -> Workspace:
    """History raw K / V with planted blocks plus one step's queries (recipe 1-4)."""
    n_blocks = wl.n_blocks if n_blocks is None else n_blocks
    gen = _gen(seed, device)
    d = wl.head_dim
    if wl.n_topics > 1:
        u = unit_vectors(wl.n_topics, d, gen, device)
    else:
        u = unit_vectors(1, d, gen, device)[0]
    planted = planted_blocks(wl, n_blocks, gen)
    ws = Workspace(wl=wl, u=u, planted=planted)
    if wl.n_topics > 1:
        ws.topic_of = torch.randint(0, wl.n_topics, (planted.numel(),), generator=gen,
                                    device=device)
    if with_kv:
        shape = (n_blocks, wl.n_layers, wl.n_kv_heads, BLOCK_TOKENS, d)
        kvd = torch_dtype(wl.kv_dtype)
        raw = _randn(shape, gen, device, scale=wl.k_std, out_dtype=kvd)
        if planted.numel():
            if wl.n_topics > 1:
                shift = (wl.k_shift * wl.k_std) * u[ws.topic_of]          # [P, d]
                shift = shift[:, None, None, None, :]
            else:
                shift = (wl.k_shift * wl.k_std) * u
            sel = _from_storage(raw[planted]) + shift
            raw[planted] = _to_storage(sel, raw.dtype)
        ws.raw_k = raw
        ws.v = _randn(shape, gen, device, scale=wl.k_std, out_dtype=kvd)
    if with_q:
        ws.q = make_queries(wl, gen, device, u if wl.n_topics == 1 else None)
    return ws


def make_queries(wl: Workload, gen, device, direction: torch.Tensor | None,
                 topic_dirs: torch.Tensor | None = None) -> torch.Tensor:
    """RoPE-free queries ``[L][M_q][H][d]``: N(0,1) + q_shift along a direction.

    ``direction`` shifts every query along one vector; ``topic_dirs`` ([M_q, d])
    gives each query its own direction (churn steps)."""
    q = torch.randn(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim, generator=gen,
                    device=device, dtype=torch.float32)
    if topic_dirs is not None:
        q += wl.q_shift * topic_dirs[None, :, None, :]
    elif direction is not None:
        q += wl.q_shift * direction
    return q.to(torch_dtype(wl.q_dtype))


def make_index_direct(wl: Workload, seed: int = 0, device="cpu",
                      n_blocks: int | None = None) -> Workspace:
    """Mean-K index drawn directly, ``[L][G][N][d]`` ~ N(0, k_std^2), planted blocks
    shifted by ``k_shift * k_std * u`` (scoring-only workload), plus queries."""
    n_blocks = wl.n_blocks if n_blocks is None else n_blocks
    gen = _gen(seed, device)
    u = unit_vectors(1, wl.head_dim, gen, device)[0]
    planted = planted_blocks(wl, n_blocks, gen)
    idx = _randn((wl.n_layers, wl.n_kv_heads, n_blocks, wl.head_dim), gen, device,
                 scale=wl.k_std, out_dtype=torch_dtype(wl.index_dtype))
    if planted.numel():
        sub = idx[:, :, planted, :].float() + (wl.k_shift * wl.k_std) * u
        idx[:, :, planted, :] = sub.to(idx.dtype)
    q = make_queries(wl, gen, device, u)
    return Workspace(wl=wl, u=u, planted=planted, index=idx, q=q)


def churn_topics(wl: Workload, seed: int, device="cpu") -> list[torch.Tensor]:
    """Active topic sets A_0..A_{steps-1}: ``topics_per_step`` topics per step, of
    which ``round(overlap * topics_per_step)`` are kept from the previous step."""
    gen = _gen(seed + 7919, "cpu")
    k = wl.topics_per_step
    keep = int(round(wl.overlap * k))
    a = torch.randperm(wl.n_topics, generator=gen)[:k]
    out = [a]
    for _ in range(1, wl.steps):
        kept = a[torch.randperm(k, generator=gen)[:keep]]
        pool = torch.tensor([t for t in range(wl.n_topics) if t not in set(a.tolist())])
        new = pool[torch.randperm(pool.numel(), generator=gen)[:k - keep]]
        a = torch.cat([kept, new])
        out.append(a)
    return [t.to(device) for t in out]


def churn_queries(wl: Workload, ws: Workspace, step: int, topics: torch.Tensor,
                  seed: int, device="cpu") -> torch.Tensor:
    """Queries of churn step ``step``: query m is shifted along u_{A_t[m mod k]}."""
    gen = _gen(seed * 1000 + 17 + step, device)
    dirs = ws.u[topics[torch.arange(wl.n_queries, device=topics.device) % topics.numel()]]
    return make_queries(wl, gen, device, None, topic_dirs=dirs.to(device))
