"""Shared pieces of the GPU parity tests: test-size workloads, the parity rules
and comparisons against the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle.kvmem as ora
from paged_kv_cache_meank_gb300 import configs

# bf16, d = 128, the 27B-class query rows per KV head (32 queries x GQA 6 = 192),
# several scoring chunks with a ragged tail, 60-slot view
MID = configs.Workload(
    name="mid-bf16-d128", n_layers=4, n_kv_heads=2, n_q_heads=12, head_dim=128,
    rope_theta=1e6, kv_dtype="bf16", index_dtype="bf16", q_dtype="bf16", n_blocks=300,
    n_queries=32, sink_blocks=4, recent_blocks=8, view_blocks=60, planted_frac=0.05,
    k_std=1.0 / 128 ** 0.5)

# bf16, d = 64, GQA 2, 20 queries (40 rows), odd block count
MID64 = configs.Workload(
    name="mid-bf16-d64", n_layers=3, n_kv_heads=4, n_q_heads=8, head_dim=64, rope_theta=1e4,
    kv_dtype="bf16", index_dtype="bf16", q_dtype="bf16", n_blocks=257, n_queries=20,
    sink_blocks=2, recent_blocks=3, view_blocks=40, planted_frac=0.04, k_std=0.125)

# float32 K with a float32 index but bf16 queries
MIXED = configs.Workload(
    name="mixed-f32kv-bf16q", n_layers=2, n_kv_heads=1, n_q_heads=4, head_dim=128,
    rope_theta=1e6, kv_dtype="f32", index_dtype="f32", q_dtype="bf16", n_blocks=150,
    n_queries=8, sink_blocks=1, recent_blocks=2, view_blocks=20, planted_frac=0.05)

# 8-bit (e4m3) K / V pages with a bf16 index, d = 128
FP8 = MID.with_(name="mid-e4m3-d128", kv_dtype="e4m3", n_blocks=211)

SMALL = [configs.TINY, MID, MID64, MIXED, FP8]

REL_SCORE = 1e-4   # relative tolerance on R_b


def to_np(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "e4m3":
        return t.view(torch.uint8).numpy().copy()
    return t.float().numpy().copy()


def from_np(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16).to(device)
    if dtype == "e4m3":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    """Monotone integer image of bf16 bit patterns (adjacent values differ by 1)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF) - 1, b + 0x8000 - 1 + 1)


def e4m3_ordered(bits: np.ndarray) -> np.ndarray:
    """Monotone integer image of e4m3 bit patterns (+0 and -0 both map to 0)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x80, -(b & 0x7F), b)


def assert_storage_close(gpu: np.ndarray, ref: np.ndarray, dtype: str, what: str,
                         f32_pair_ulps: float = 2.0):
    """K-type outputs: bf16 and e4m3 within 1 ulp of the reference rounding;
    float32 within ``f32_pair_ulps`` ulps of the rotate-half pair's magnitude."""
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if dtype in ("bf16", "e4m3"):
        order = bf16_ordered if dtype == "bf16" else e4m3_ordered
        d = np.abs(order(gpu) - order(ref))
        bad = int((d > 1).sum())
        assert bad == 0, f"{what}: {bad} elements beyond 1 {dtype} ulp (max {d.max()})"
        return float((d == 0).mean())
    h = ref.shape[-1] // 2
    mag = np.maximum(np.abs(ref[..., :h]), np.abs(ref[..., h:]))
    mag = np.concatenate([mag, mag], axis=-1)
    tol = f32_pair_ulps * np.spacing(np.maximum(mag, 1e-30).astype(np.float32)).astype(np.float64)
    err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    bad = int((err > tol).sum())
    assert bad == 0, f"{what}: {bad} elements beyond {f32_pair_ulps} pair ulps"
    return float((gpu == ref).mean())


def assert_meank_close(gpu: np.ndarray, ref64: np.ndarray, dtype: str, k_rms: float, what: str,
                       k_max: float | None = None):
    """Mean-K against the float64 mean.

    The kernel un-rotates in float32 (one rounding per product and sum) and
    sums 32 float32 terms before one rounding to the index dtype, so its error
    before that rounding is at most (2 + 31) * 2^-24 * max|K| in absolute terms.
    bf16: within 1 ulp of the reference plus that bound (the bound only matters
    for means that nearly cancel); float32: within 1e-6 * rms(K) absolute."""
    if dtype == "bf16":
        g = ora.bf16_to_f32(gpu).astype(np.float64)
        mag = np.abs(ref64)
        ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.maximum(mag, 1e-300))) - 7), 0.0)
        acc = 33 * 2.0 ** -24 * (k_max if k_max is not None else 8 * k_rms)
        err = np.abs(g - ref64)
        bad = err > ulp * (1 + 1e-9) + acc
        assert not bad.any(), f"{what}: {int(bad.sum())} Mean-K entries beyond 1 bf16 ulp + {acc:.2g}"
    else:
        err = np.abs(gpu.astype(np.float64) - ref64)
        assert err.max() <= 1e-6 * k_rms, f"{what}: Mean-K error {err.max()}"


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    rel = np.abs(gpu.astype(np.float64) - ref) / np.abs(ref)
    assert rel.max() <= REL_SCORE, f"{what}: max relative score error {rel.max():.3g}"
    return float(rel.max())


def check_selection(gpu_sel: np.ndarray, R: np.ndarray, S: int, W: int, V: int,
                    what: str = "") -> int:
    """The selection rule with the near-tie band: every candidate with
    R > T(1+1e-4) must be selected, none with R < T(1-1e-4); reserved blocks
    always; ascending; exactly min(N, V) ids.  Returns how many candidates fell
    inside the band."""
    N = len(R)
    sel = [int(x) for x in gpu_sel]
    assert sel == sorted(set(sel)), f"{what}: not strictly ascending"
    if N <= V:
        assert sel == list(range(N)), what
        return 0
    assert len(sel) == V, (what, len(sel), V)
    reserved = set(range(S)) | set(range(N - W, N))
    assert reserved <= set(sel), f"{what}: reserved block missing"
    T = ora.kth_boundary(R, S, W, V)
    chosen = set(sel) - reserved
    hi, lo = T * (1 + REL_SCORE), T * (1 - REL_SCORE)
    band = 0
    for b in range(N):
        if b in reserved:
            continue
        if R[b] > hi:
            assert b in chosen, f"{what}: block {b} (R={R[b]:.8g} > T={T:.8g}) not selected"
        elif R[b] < lo:
            assert b not in chosen, f"{what}: block {b} (R={R[b]:.8g} < T={T:.8g}) selected"
        else:
            band += 1
    return band
