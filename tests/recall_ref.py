"""Composes the CPU oracle's steps into one recall step (test helper).

Inputs come from ``paged_kv_cache_meank_gb300.workload`` (random draws only);
every computed value here comes from ``oracle``.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.kvmem as ora


def to_np(t: torch.Tensor, dtype: str) -> np.ndarray:
    """A CPU tensor as the oracle's storage form (uint16 bf16 bits or float32)."""
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "e4m3":
        return t.view(torch.uint8).numpy().copy()
    return t.float().numpy().copy()


def from_np(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    if dtype == "e4m3":
        return torch.from_numpy(np.asarray(a, dtype=np.uint8).copy())
    return torch.from_numpy(np.asarray(a, dtype=np.float32).copy())


def prefill_k_pages(raw_k: np.ndarray, kv_dtype: str, theta: float, first_block: int = 0):
    """K as a model's prefill writes it: raw K rotated at original positions in
    float32 from the float32 tables, rounded to the storage dtype."""
    r32 = ora.as_f32(raw_k, kv_dtype)
    n, L, G, B, d = r32.shape
    pos = ora.block_positions(np.arange(first_block, first_block + n))
    out = np.empty_like(r32)
    for i in range(n):
        c, s = ora.cos_sin_f32(pos[i], d, theta)
        out[i] = ora.rope_f32(r32[i], c, s)
    return ora.round_to(out, kv_dtype)


def recall(wl, k_pages, v, q, n_blocks=None):
    """One oracle recall step over a history given as prefill K pages.
    Returns a dict with index (f64), raw_k (storage), R, sel, view K/V."""
    n_blocks = k_pages.shape[0] if n_blocks is None else n_blocks
    index = ora.meank(k_pages[:n_blocks], wl.kv_dtype, 0, wl.rope_theta)
    rk = ora.raw_k(k_pages[:n_blocks], wl.kv_dtype, 0, wl.rope_theta)
    q64 = ora.as_f64(q, wl.q_dtype)
    index_stored = ora.as_f64(ora.round_to(index.astype(np.float32), wl.index_dtype),
                              wl.index_dtype)
    R = ora.block_relevance(q64, index_stored, n_blocks)
    sel = ora.select_blocks(R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)
    vk = ora.view_k(rk[sel], wl.kv_dtype, wl.rope_theta)
    vv = v[sel]
    return dict(index=index, index_stored=index_stored, raw_k=rk, R=R, sel=sel,
                view_k=vk, view_v=vv)
