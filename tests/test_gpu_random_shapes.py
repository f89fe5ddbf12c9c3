"""Parity over seeded random shapes, through the C ABI: Mean-K build, Eq. (10)
scoring with selection, and view assembly, each against the CPU oracle.

The fixed-shape tests pick the workloads' own shapes and their edges; this
sweep draws the rest of the space the library accepts: layer and KV-head
counts, GQA ratios, head dims 64 and 128, f32 / bf16 / e4m3 pages, f32 and
bf16 index and queries, ragged history lengths (some above 16384 blocks,
where the selection runs on many CTAs), sink / recent / view budgets that
may exceed the history, both candidate-set readings, and both scoring
variants.  Inputs come from the seeded generator; every expected value comes
from the oracle (the index scored here is the oracle's Mean-K rounded to the
index dtype, the view is rotated from the oracle's raw K).
"""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import (assert_meank_close, assert_scores_close, assert_storage_close,
                         check_selection, from_np, to_np)
from paged_kv_cache_meank_gb300 import configs
from recall_ref import prefill_k_pages
from step_helpers import run_steps

pytestmark = pytest.mark.gpu


def _cases(seed: int, n_short: int, n_long: int):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_short + n_long):
        long = i >= n_short
        d = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 3, 4, 8]))
        r = int(rng.choice([1, 2, 3, 4, 6, 8]))
        L = 1 if long else int(rng.integers(1, 5))
        if long:
            G, d = 1, 64
        nq = int(rng.integers(1, min(40, 256 // r) + 1))
        N = int(rng.integers(16385, 20000)) if long else int(rng.integers(1, 2500))
        if not long:
            # at most about 30M K elements, so the float64 oracle stays quick
            N = max(1, min(N, 30_000_000 // (L * G * 32 * d)))
        S = int(rng.integers(0, 6))
        W = int(rng.integers(0, 12))
        V = S + W + int(rng.integers(1, 150))
        kv = str(rng.choice(["f32", "bf16", "e4m3"]))
        idx = str(rng.choice(["f32", "bf16", "bf16"]))
        qd = str(rng.choice(["f32", "bf16", "bf16"]))
        theta = float(rng.choice([1e4, 1e6]))
        mode = int(rng.integers(0, 2)) if N > S + W + 1 else 0
        wl = configs.Workload(
            name=f"rand{i}-L{L}G{G}r{r}d{d}-{kv}-{idx}-{qd}-N{N}-S{S}W{W}V{V}-m{mode}",
            n_layers=L, n_kv_heads=G, n_q_heads=G * r, head_dim=d, rope_theta=theta,
            kv_dtype=kv, index_dtype=idx, q_dtype=qd, n_blocks=N, n_queries=nq,
            sink_blocks=S, recent_blocks=W, view_blocks=V, planted_frac=0.03,
            k_std=1.0 / d ** 0.5)
        out.append((wl, mode, int(rng.integers(0, 1 << 30))))
    return out


CASES = _cases(20261202, n_short=30, n_long=4)


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return kvm


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_random_shape_recall(kvm, case):
    from paged_kv_cache_meank_gb300 import workload
    wl, mode, seed = case
    N, V, S, W = wl.n_blocks, wl.view_blocks, wl.sink_blocks, wl.recent_blocks
    ws = workload.make_workspace(wl, seed=seed)
    raw = to_np(ws.raw_k, wl.kv_dtype)
    kp = prefill_k_pages(raw, wl.kv_dtype, wl.rope_theta)

    # (a) Mean-K build with raw K out
    ctx0 = kvm.Context(kvm.config_for(wl, candidate_mode=mode))
    index = torch.zeros(ctx0.index_shape(), dtype=ctx0.index_dtype, device="cuda")
    raw_out = torch.zeros(ctx0.block_shape(N), dtype=ctx0.kv_dtype, device="cuda")
    ctx0.build_index(from_np(kp, wl.kv_dtype), 0, N, index, raw_out)
    ctx0.sync()
    mean64 = ora.meank(kp, wl.kv_dtype, 0, wl.rope_theta)
    rms = float(np.sqrt(np.mean(ora.as_f64(raw, wl.kv_dtype) ** 2)))
    kmax = float(np.abs(ora.as_f64(kp, wl.kv_dtype)).max()) * 2 ** 0.5
    if wl.index_dtype == "bf16":
        assert_meank_close(to_np(index, "bf16"), mean64, "bf16", rms, wl.name, kmax)
    else:
        # float32 Mean-K: the kernel's own arithmetic bound (two roundings per
        # un-rotated term, 31 in the token sum; the division by 32 is exact)
        err = np.abs(to_np(index, "f32").astype(np.float64) - mean64)
        assert err.max() <= 33 * 2.0 ** -24 * kmax, (wl.name, float(err.max()))
    raw_ref = ora.raw_k(kp, wl.kv_dtype, 0, wl.rope_theta)
    assert_storage_close(to_np(raw_out, wl.kv_dtype), raw_ref, wl.kv_dtype, wl.name + " raw K")

    # (b) scoring + selection on the oracle's rounded index, both variants
    idx_np = ora.round_to(mean64.astype(np.float32), wl.index_dtype)
    q64 = ora.as_f64(to_np(ws.q, wl.q_dtype), wl.q_dtype)
    i64 = ora.as_f64(idx_np, wl.index_dtype)
    R = (ora.block_relevance_excl(q64, i64, N, S, W) if mode == 1
         else ora.block_relevance(q64, i64, N))
    idx_d = from_np(idx_np, wl.index_dtype)
    q_d = ws.q.to("cuda")
    sels = []
    for variant in (0, 1):
        ctx = kvm.Context(kvm.config_for(wl, candidate_mode=mode, score_variant=variant))
        scores = torch.empty(N, dtype=torch.float32, device="cuda")
        sel = torch.full((V,), -1, dtype=torch.int32, device="cuda")
        n_sel = ctx.score_select(q_d, wl.n_queries, idx_d, N, scores, sel)
        ctx.sync()
        assert n_sel == min(N, V)
        got = scores.cpu().numpy()
        if mode == 1:
            lo, hi = ora.candidate_range(N, S, W)
            assert np.all(got[:lo] == 0) and np.all(got[hi:] == 0), wl.name
            assert_scores_close(got[lo:hi], R[lo:hi], f"{wl.name} v{variant}")
        else:
            assert_scores_close(got, R, f"{wl.name} v{variant}")
        sel_np = sel.cpu().numpy()[:n_sel]
        band = check_selection(sel_np, R, S, W, V, f"{wl.name} v{variant}")
        if band == 0:
            assert np.array_equal(sel_np, ora.select_blocks(R, S, W, V)), wl.name
        sels.append(sel_np)

    # (c) view assembly of the GPU's own selection into permuted pages, from
    # the oracle's raw K
    ids = sels[0]
    n_sel = len(ids)
    perm = np.random.default_rng(seed).permutation(n_sel + 3)[:n_sel].astype(np.int32)
    kp_out = torch.full(ctx0.block_shape(n_sel + 3), 3.0, device="cuda").to(ctx0.kv_dtype)
    vp_out = torch.full_like(kp_out, 0)
    ctx0.assemble_view(torch.from_numpy(ids.astype(np.int32)).cuda(),
                       torch.from_numpy(perm).cuda(), n_sel, from_np(raw_ref, wl.kv_dtype),
                       ws.v.to("cuda"), kp_out, vp_out)
    ctx0.sync()
    ref_k = ora.view_k(raw_ref[ids], wl.kv_dtype, wl.rope_theta)
    assert_storage_close(to_np(kp_out, wl.kv_dtype)[perm], ref_k, wl.kv_dtype,
                         wl.name + " view K")
    assert np.array_equal(to_np(vp_out, wl.kv_dtype)[perm], to_np(ws.v, wl.kv_dtype)[ids])


def _step_cases(seed: int, n: int):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        G = int(rng.choice([1, 2, 4]))
        r = int(rng.choice([1, 2, 3, 6]))
        L = int(rng.integers(1, 4))
        kv = str(rng.choice(["f32", "bf16", "e4m3"]))
        idx = str(rng.choice(["f32", "bf16", "bf16"]))
        qd = str(rng.choice(["f32", "bf16", "bf16"]))
        S = int(rng.integers(0, 5))
        W = int(rng.integers(0, 9))
        V = S + W + int(rng.integers(1, 80))
        n_cap = max(2, min(1500, 20_000_000 // (L * G * 32 * d)))
        ns = [int(rng.integers(1, n_cap))]
        for _ in range(3):   # the history grows, or shrinks (possibly below V)
            ns.append(int(np.clip(ns[-1] + rng.integers(-ns[-1] // 2 - 1, 200), 1, n_cap)))
        repo_host = bool(rng.integers(0, 2))
        h2d_mode = int(rng.integers(0, 2)) if repo_host else 0
        index_host = bool(rng.integers(0, 2))
        spill = int(rng.integers(0, 2)) if index_host else 0
        q_order = [int(x) for x in rng.integers(0, 3, size=len(ns))]
        wl = configs.Workload(
            name=(f"steps{i}-L{L}G{G}r{r}d{d}-{kv}-{idx}-{qd}-S{S}W{W}V{V}-"
                  f"N{'_'.join(map(str, ns))}-{'host' if repo_host else 'dev'}{h2d_mode}"
                  f"-{'hidx' if index_host else 'didx'}{spill}"),
            n_layers=L, n_kv_heads=G, n_q_heads=G * r, head_dim=d,
            rope_theta=float(rng.choice([1e4, 1e6])), kv_dtype=kv, index_dtype=idx,
            q_dtype=qd, n_blocks=max(ns), n_queries=int(rng.integers(1, min(24, 256 // r) + 1)),
            sink_blocks=S, recent_blocks=W, view_blocks=V, planted_frac=0.03,
            k_std=1.0 / d ** 0.5)
        out.append((wl, ns, repo_host, h2d_mode, index_host, spill, q_order,
                    int(rng.integers(0, 1 << 30))))
    return out


STEP_CASES = _step_cases(20261203, 20)


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: c[0].name)
def test_random_shape_steps(kvm, case):
    """kvm_step over four steps on a random shape: scores, selection, the
    oracle's delta working set applied to the GPU's selection (page table,
    hits, misses, re-RoPE count, H2D bytes) and the materialised view."""
    from paged_kv_cache_meank_gb300 import workload
    wl, ns, repo_host, h2d_mode, index_host, spill, q_order, seed = case
    g = torch.Generator().manual_seed(seed)
    u = workload.unit_vectors(3, wl.head_dim, g, "cpu")
    qs = [workload.make_queries(wl, g, "cpu", u[k]) for k in range(3)]
    hist = run_steps(kvm, wl, repo_host, index_host, [qs[k] for k in q_order], ns,
                      h2d_mode=h2d_mode, index_spill=spill)
    assert hist[0]["hits"] == 0 and hist[0]["misses"] == min(ns[0], wl.view_blocks)
    for a in range(1, len(ns)):
        if q_order[a] == q_order[a - 1] and ns[a] == ns[a - 1]:
            # the same queries over the same history: nothing moves
            assert hist[a]["misses"] == 0 and hist[a]["reroped"] == 0
