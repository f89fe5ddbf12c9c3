"""Per-call parity of the CUDA path against the CPU oracle, through the C ABI.

Sizes span several scoring chunks, a ragged tail, both head dims and both
element types.  Inputs come from the seeded generator (raw K / V, queries,
directly drawn Mean-K) and from the oracle (K rotated at original positions,
as a prefill writes it); nothing the oracle consumes comes from the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import (MID, MID64, SMALL, assert_meank_close, assert_scores_close,
                         assert_storage_close, check_selection, from_np, to_np)
from recall_ref import prefill_k_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return kvm


def _ctx(kvm, wl, **kw):
    return kvm.Context(kvm.config_for(wl, **kw))


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_build_index(kvm, wl):
    from paged_kv_cache_meank_gb300 import workload
    ws = workload.make_workspace(wl, seed=1, with_q=False)
    raw = to_np(ws.raw_k, wl.kv_dtype)
    kp = prefill_k_pages(raw, wl.kv_dtype, wl.rope_theta)
    N = wl.n_blocks
    ctx = _ctx(kvm, wl, max_blocks=N + 5)
    kp_d = from_np(kp, wl.kv_dtype)
    index = torch.full(ctx.index_shape(), 7.0, dtype=ctx.index_dtype, device="cuda")
    raw_out = torch.zeros(ctx.block_shape(N), dtype=ctx.kv_dtype, device="cuda")
    # two incremental calls, as blocks complete during prefill
    cut = N // 3
    ctx.build_index(kp_d[:cut], 0, cut, index, raw_out[:cut])
    ctx.build_index(kp_d[cut:], cut, N - cut, index, raw_out[cut:])
    ctx.sync()
    ref = ora.meank(kp, wl.kv_dtype, 0, wl.rope_theta)
    got = to_np(index[:, :, :N], wl.index_dtype)
    rms = float(np.sqrt(np.mean(ora.as_f64(raw, wl.kv_dtype) ** 2)))
    kmax = float(np.abs(ora.as_f64(kp, wl.kv_dtype)).max()) * 2 ** 0.5
    assert_meank_close(got, ref, wl.index_dtype, rms, wl.name, kmax)
    # entries past the built range are untouched
    assert torch.all(index[:, :, N:].float() == 7.0)
    exact = assert_storage_close(to_np(raw_out, wl.kv_dtype),
                                 ora.raw_k(kp, wl.kv_dtype, 0, wl.rope_theta), wl.kv_dtype,
                                 wl.name + " raw K")
    assert exact > 0.999


@pytest.mark.parametrize("variant", [0, 1], ids=["tensor-cores", "cuda-cores"])
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_score_select(kvm, wl, variant):
    from paged_kv_cache_meank_gb300 import workload
    ws = workload.make_index_direct(wl, seed=2)
    N = wl.n_blocks
    ctx = _ctx(kvm, wl, score_variant=variant)
    index = ws.index.to("cuda")
    q = ws.q.to("cuda")
    scores = torch.empty(N, dtype=torch.float32, device="cuda")
    sel = torch.full((wl.view_blocks,), -1, dtype=torch.int32, device="cuda")
    n_sel = ctx.score_select(q, wl.n_queries, index, N, scores, sel)
    ctx.sync()
    assert n_sel == min(N, wl.view_blocks)
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, wl.q_dtype), wl.q_dtype),
                            ora.as_f64(to_np(ws.index, wl.index_dtype), wl.index_dtype), N)
    assert_scores_close(scores.cpu().numpy(), R, wl.name)
    band = check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks,
                           wl.view_blocks, wl.name)
    if band == 0:
        want = ora.select_blocks(R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)
        assert np.array_equal(sel.cpu().numpy(), want)
    # run twice: bitwise identical
    scores2, sel2 = torch.empty_like(scores), torch.empty_like(sel)
    ctx.score_select(q, wl.n_queries, index, N, scores2, sel2)
    ctx.sync()
    assert torch.equal(scores, scores2) and torch.equal(sel, sel2)


@pytest.mark.parametrize("variant", [0, 1], ids=["tensor-cores", "cuda-cores"])
def test_score_select_fewer_queries_and_ragged(kvm, variant):
    """n_queries below the configured maximum, N not a multiple of any tile."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=1237, view_blocks=100)
    ws = workload.make_index_direct(wl, seed=3)
    ctx = _ctx(kvm, wl, max_queries=wl.n_queries, score_variant=variant)
    nq = 7
    q = ws.q[:, :nq].contiguous().to("cuda")
    scores = torch.empty(wl.n_blocks, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.score_select(q, nq, ws.index.to("cuda"), wl.n_blocks, scores, sel)
    ctx.sync()
    R = ora.block_relevance(ora.as_f64(to_np(ws.q[:, :nq], "bf16"), "bf16"),
                            ora.as_f64(to_np(ws.index, "bf16"), "bf16"), wl.n_blocks)
    assert_scores_close(scores.cpu().numpy(), R, "fewer queries")
    assert abs(float(scores.double().sum()) - nq) < 1e-3 * nq
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)


@pytest.mark.parametrize("variant", [0, 1], ids=["tensor-cores", "cuda-cores"])
@pytest.mark.parametrize("loc", ["device", "host-tiled", "host-tiled-spill",
                                 "host-tiled-spill-budget"])
def test_score_select_candidates_exclude_reserved(kvm, variant, loc):
    """candidate_mode 1: the Eq. (10) softmax runs over the non-reserved blocks
    only; sink and recent blocks score exactly 0 and are still selected.  The
    host-tiled index puts the candidate range's ends inside 96-block tiles;
    with index_spill pass 2 reads the tiles pass 1 staged (all 13, or the
    last 4 under a spill budget, the first 9 crossing the link again)."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=1237, view_blocks=100)
    ws = workload.make_index_direct(wl, seed=4)
    kw = dict(score_variant=variant, candidate_mode=1)
    index = ws.index.to("cuda")
    if loc.startswith("host-tiled"):
        kw["index_location"] = kvm.KVM_HOST_PINNED
        kw["index_spill"] = int("spill" in loc)
        kw["spill_tiles"] = 4 if loc.endswith("budget") else 0
        index = ws.index.pin_memory()
    cfg = kvm.config_for(wl, **kw)
    if loc.startswith("host-tiled"):
        cfg.tile_blocks = 96
    ctx = kvm.Context(cfg)
    N, S, W = wl.n_blocks, wl.sink_blocks, wl.recent_blocks
    scores = torch.full((N,), 5.0, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.score_select(ws.q.cuda(), wl.n_queries, index, N, scores, sel)
    ctx.sync()
    got = scores.cpu().double().numpy()
    R = ora.block_relevance_excl(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                                 ora.as_f64(to_np(ws.index, "bf16"), "bf16"), N, S, W)
    assert np.all(got[:S] == 0) and np.all(got[N - W:] == 0)
    assert_scores_close(got[S:N - W], R[S:N - W], "candidates only")
    assert abs(got.sum() - wl.n_queries) < 1e-3 * wl.n_queries
    check_selection(sel.cpu().numpy(), R, S, W, wl.view_blocks, "candidates only")


@pytest.mark.parametrize("candidate_mode", [0, 1])
def test_host_tiled_results_do_not_depend_on_the_spill(kvm, candidate_mode):
    """A host-resident index in 96-block tiles (13 tiles, the last one ragged):
    streamed twice, kept whole, or kept up to a budget of 1, 4 or 12 tiles
    (pass 2 then scores the kept tiles first), the scores and the selection
    are bit-identical; the first also matches the oracle."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=1237, view_blocks=100)
    ws = workload.make_index_direct(wl, seed=8)
    index = ws.index.pin_memory()
    q = ws.q.cuda()
    N = wl.n_blocks
    got = []
    for spill, m in [(0, 0), (1, 0), (1, 1), (1, 4), (1, 12)]:
        cfg = kvm.config_for(wl, index_location=kvm.KVM_HOST_PINNED, index_spill=spill,
                             spill_tiles=m, candidate_mode=candidate_mode)
        cfg.tile_blocks = 96
        ctx = kvm.Context(cfg)
        scores = torch.empty(N, device="cuda")
        sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
        for _ in range(2):          # the second call reuses the kept tiles' buffers
            ctx.score_select(q, wl.n_queries, index, N, scores, sel)
        ctx.sync()
        got.append((scores.cpu(), sel.cpu()))
        ctx.close()
    for sc, se in got[1:]:
        assert torch.equal(sc, got[0][0]) and torch.equal(se, got[0][1])
    q64 = ora.as_f64(to_np(ws.q, "bf16"), "bf16")
    i64 = ora.as_f64(to_np(ws.index, "bf16"), "bf16")
    S, W = wl.sink_blocks, wl.recent_blocks
    R = (ora.block_relevance_excl(q64, i64, N, S, W) if candidate_mode
         else ora.block_relevance(q64, i64, N))
    lo, hi = (S, N - W) if candidate_mode else (0, N)
    assert_scores_close(got[0][0].double().numpy()[lo:hi], R[lo:hi], "host tiles")
    check_selection(got[0][1].numpy(), R, S, W, wl.view_blocks, "host tiles")


@pytest.mark.parametrize("loc", ["device", "host-tiled"])
@pytest.mark.parametrize("nth", [1, 2], ids=["pass1", "pass2"])
def test_bounded_wait_runs_out_and_context_recovers(kvm, nth, loc):
    """A tensor-core pass whose TMA producer stays idle (a barrier that nothing
    completes): its bounded waits run out after about a second, the kernel
    winds down and frees its TMEM, kvm_sync reports KVM_ERR_TIMEOUT, and the
    next call on the same context matches the oracle."""
    import time
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    ws = workload.make_index_direct(wl, seed=6)
    kw = {}
    index = ws.index.to("cuda")
    if loc == "host-tiled":
        kw["index_location"] = kvm.KVM_HOST_PINNED
        index = ws.index.pin_memory()
    cfg = kvm.config_for(wl, **kw)
    if loc == "host-tiled":
        cfg.tile_blocks = 128
    ctx = kvm.Context(cfg)
    N = wl.n_blocks
    q = ws.q.cuda()
    scores = torch.empty(N, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    # launches of the host-tiled path: pass 1 over the 3 tiles, then pass 2
    ctx.debug_inject(3, nth if loc == "device" else 1 + 3 * (nth - 1))
    t0 = time.monotonic()
    ctx.score_select(q, wl.n_queries, index, N, scores, sel)
    with pytest.raises(kvm.KvmError) as ei:
        ctx.sync()
    assert ei.value.name == "KVM_ERR_TIMEOUT"
    assert time.monotonic() - t0 < 30.0
    s = sel.cpu().numpy()
    assert np.all((s >= 0) & (s < N))
    # the same context, the next call: parity
    ctx.score_select(q, wl.n_queries, index, N, scores, sel)
    ctx.sync()
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                            ora.as_f64(to_np(ws.index, "bf16"), "bf16"), N)
    assert_scores_close(scores.cpu().numpy(), R, "after a timed-out pass")
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)


@pytest.mark.parametrize("n_queries", [21, 32, 40, 42], ids=lambda n: f"rows{n * 6}")
def test_score_select_query_row_tilings(kvm, n_queries):
    """Query rows per KV head across the tensor-core tilings: one M = 128 tile
    (126 rows), the duplicated second tile (129..192 rows) and two full tiles
    (240, 252 rows)."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=517, view_blocks=50, n_queries=n_queries)
    ws = workload.make_index_direct(wl, seed=30 + n_queries)
    ctx = _ctx(kvm, wl)
    scores = torch.empty(wl.n_blocks, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.score_select(ws.q.cuda(), n_queries, ws.index.cuda(), wl.n_blocks, scores, sel)
    ctx.sync()
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                            ora.as_f64(to_np(ws.index, "bf16"), "bf16"), wl.n_blocks)
    assert_scores_close(scores.cpu().numpy(), R, f"{n_queries * 6} rows")
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)


@pytest.mark.parametrize("n_q_heads,n_queries", [(16, 32), (16, 16), (2, 129), (2, 1), (4, 3)],
                         ids=["rows256", "rows128", "rows129", "rows1", "rows6"])
def test_score_select_query_row_extremes(kvm, n_q_heads, n_queries):
    """The ends of the tensor-core row tilings with other GQA ratios: the
    largest count (256 rows, two full M = 128 tiles), exactly one tile (128),
    one row past it (129, the duplicated second tile at its smallest), a single
    row (MMA N = 16 with 15 padding columns) and 6 rows."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=389, view_blocks=40, n_q_heads=n_q_heads, n_queries=n_queries)
    ws = workload.make_index_direct(wl, seed=60 + n_queries)
    ctx = _ctx(kvm, wl)
    scores = torch.empty(wl.n_blocks, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.score_select(ws.q.cuda(), n_queries, ws.index.cuda(), wl.n_blocks, scores, sel)
    ctx.sync()
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                            ora.as_f64(to_np(ws.index, "bf16"), "bf16"), wl.n_blocks)
    rows = n_queries * (n_q_heads // wl.n_kv_heads)
    assert_scores_close(scores.cpu().numpy(), R, f"{rows} rows")
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)


def test_select_ties_and_small_histories(kvm):
    """Equal Mean-K everywhere: all scores tie and the lowest ids win; histories
    of N <= V_b select everything; N = V_b + 1 leaves out exactly one block."""
    wl = MID64
    ctx = _ctx(kvm, wl)
    q = torch.randn(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim,
                    device="cuda").to(torch.bfloat16)
    for N in (1, 5, wl.view_blocks, wl.view_blocks + 1, 200):
        index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
        index[:, :, :N] = 0.25
        scores = torch.empty(N, device="cuda")
        sel = torch.full((wl.view_blocks,), -1, dtype=torch.int32, device="cuda")
        n_sel = ctx.score_select(q, wl.n_queries, index, N, scores, sel)
        ctx.sync()
        got = sel[:n_sel].cpu().numpy()
        want = ora.select_blocks(np.full(N, 1.0 / N), wl.sink_blocks, wl.recent_blocks,
                                 wl.view_blocks)
        assert np.array_equal(got, want), (N, got, want)
        assert torch.allclose(scores, torch.full_like(scores, wl.n_queries / N), rtol=1e-5)


@pytest.mark.parametrize("variant", [0, 1], ids=["tensor-cores", "cuda-cores"])
def test_empty_and_degenerate_inputs(kvm, variant):
    """Empty calls are no-ops or rejected on the host; an empty candidate set
    (every block reserved) scores 0 everywhere and selects every block."""
    wl = MID
    ctx = _ctx(kvm, wl, score_variant=variant)
    q = torch.randn(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim,
                    device="cuda").to(torch.bfloat16)
    index = torch.full(ctx.index_shape(), 0.5, dtype=torch.bfloat16, device="cuda")
    before = index.clone()
    kp = torch.ones(ctx.block_shape(1), dtype=torch.bfloat16, device="cuda")
    ctx.build_index(kp, 3, 0, index)                     # zero blocks: nothing written
    pages = torch.full(ctx.block_shape(2), 7.0, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(2, dtype=torch.int32, device="cuda")
    ctx.assemble_view(ids, None, 0, kp, None, pages, None)   # empty view: nothing written
    ctx.sync()
    assert torch.equal(index, before)
    assert bool((pages == 7.0).all())
    scores = torch.empty(wl.n_blocks, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    for nq, nb in ((wl.n_queries, 0), (0, wl.n_blocks)):
        with pytest.raises(kvm.KvmError) as ei:
            ctx.score_select(q, nq, index, nb, scores, sel)
        assert ei.value.name == "KVM_ERR_INVALID_ARG"
    S, W = wl.sink_blocks, wl.recent_blocks
    cx = _ctx(kvm, wl, score_variant=variant, candidate_mode=1)
    for N in (1, S + W - 1, S + W):
        scores.fill_(3.0)
        sel.fill_(-1)
        n_sel = cx.score_select(q, wl.n_queries, index, N, scores, sel)
        cx.sync()
        assert n_sel == N
        assert bool((scores[:N] == 0).all()), N
        assert np.array_equal(sel[:N].cpu().numpy(), np.arange(N)), N
    ctx.sync()


def test_two_host_threads_two_contexts(kvm):
    """Two host threads, each with its own context and stream, score, select
    and assemble at the same time (ctypes releases the GIL around the calls);
    each gets exactly what the same calls return one after the other."""
    import threading
    from paged_kv_cache_meank_gb300 import workload
    wls = [MID.with_(n_blocks=700, view_blocks=60), MID64.with_(n_blocks=20000, view_blocks=50)]
    inputs = []
    for i, wl in enumerate(wls):
        ws = workload.make_index_direct(wl, seed=80 + i)
        raw = torch.randn(wl.n_blocks, wl.n_layers, wl.n_kv_heads, 32, wl.head_dim,
                          device="cuda", generator=torch.Generator("cuda").manual_seed(90 + i))
        inputs.append((wl, ws.q.cuda(), ws.index.cuda(), raw.to(torch.bfloat16)))

    def run(i, out, stream):
        wl, q, index, raw = inputs[i]
        ctx = kvm.Context(kvm.config_for(wl), stream=stream)
        scores = torch.empty(wl.n_blocks, device="cuda")
        sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
        pages = torch.empty(ctx.block_shape(wl.view_blocks), dtype=torch.bfloat16, device="cuda")
        for _ in range(5):
            ctx.score_select(q, wl.n_queries, index, wl.n_blocks, scores, sel, stream=stream)
            ctx.assemble_view(sel, None, wl.view_blocks, raw, None, pages, None, stream=stream)
        ctx.sync(stream)
        out[i] = (scores.cpu(), sel.cpu(), pages.cpu())
        ctx.close()

    seq = {}
    for i in range(2):
        run(i, seq, torch.cuda.Stream())
    par = {}
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ts = [threading.Thread(target=run, args=(i, par, streams[i])) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    for i in range(2):
        for a, b in zip(seq[i], par[i]):
            assert torch.equal(a, b), i


@pytest.mark.parametrize("N", [389, 20000], ids=["one-cta", "many-cta"])
@pytest.mark.parametrize("S,W,V", [(0, 0, 40), (0, 8, 40), (4, 0, 40), (4, 8, 13), (0, 0, 1)],
                         ids=["topk-only", "no-sink", "no-recent", "k1", "k1-no-reserved"])
def test_select_budget_edges(kvm, N, S, W, V):
    """Budgets at their edges -- no sink blocks, no recent blocks, a top-k of one
    -- through both select paths, against the oracle's Eq. (10) and the band
    rule."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=N, sink_blocks=S, recent_blocks=W, view_blocks=V)
    ws = workload.make_index_direct(wl, seed=70 + S + W + V)
    ctx = _ctx(kvm, wl)
    scores = torch.empty(N, device="cuda")
    sel = torch.full((V,), -1, dtype=torch.int32, device="cuda")
    n_sel = ctx.score_select(ws.q.cuda(), wl.n_queries, ws.index.cuda(), N, scores, sel)
    ctx.sync()
    assert n_sel == V
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                            ora.as_f64(to_np(ws.index, "bf16"), "bf16"), N)
    assert_scores_close(scores.cpu().numpy(), R, f"S={S} W={W} V={V}")
    check_selection(sel.cpu().numpy(), R, S, W, V, f"S={S} W={W} V={V}")
    # and exactly the oracle's selection over the GPU's own scores
    want = ora.select_blocks(scores.cpu().double().numpy(), S, W, V)
    assert np.array_equal(sel.cpu().numpy(), want)


@pytest.mark.parametrize("pattern", ["random", "uniform", "classes"])
@pytest.mark.parametrize("N", [16384, 40000, 100003])
def test_select_long_histories_exact(kvm, N, pattern):
    """Histories of 16384 blocks and more take the many-CTA select.  Its ids
    must equal the oracle's selection over the oracle's scores, bit for bit,
    with large tie groups that cross segment boundaries: all blocks equal
    ("uniform"), or three exact score levels with the cut inside a tie group
    ("classes": every 20th block high, the next one middle).  Random scores
    follow the near-tie band rule, and are exact when no candidate is in it."""
    wl = MID.with_(n_blocks=N, view_blocks=3000)
    ctx = _ctx(kvm, wl, max_positions=wl.view_blocks * 32)
    L, nq, H, d = wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim
    g = torch.Generator(device="cuda").manual_seed(N)
    u = torch.randn(d, device="cuda", generator=g)
    u = u / u.norm()
    if pattern == "random":
        q = torch.randn(L, nq, H, d, device="cuda", generator=g).to(torch.bfloat16)
        index = (torch.randn(ctx.index_shape(), device="cuda", generator=g) * 0.3).to(
            torch.bfloat16)
    else:
        q = (u * 4.0).expand(L, nq, H, d).contiguous().to(torch.bfloat16)
        index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
        if pattern == "uniform":
            index[:, :, :N] = (u * 0.5).to(torch.bfloat16)
        else:
            b = torch.arange(N, device="cuda")
            level = torch.where(b % 20 == 0, 1.0, torch.where(b % 20 == 1, 0.5, 0.0))
            index[:, :, :N] = (level[:, None] * u[None, :]).to(torch.bfloat16)
    scores = torch.empty(N, device="cuda")
    sel = torch.full((wl.view_blocks,), -1, dtype=torch.int32, device="cuda")
    n_sel = ctx.score_select(q, nq, index, N, scores, sel)
    ctx.sync()
    assert n_sel == wl.view_blocks
    s_np = scores.cpu().numpy().astype(np.float64)
    R = ora.block_relevance(ora.as_f64(to_np(q.cpu(), "bf16"), "bf16"),
                            ora.as_f64(to_np(index[:, :, :N].cpu(), "bf16"), "bf16"), N)
    assert_scores_close(s_np, R, f"long history {pattern}")
    g_sel = sel.cpu().numpy()
    want = ora.select_blocks(R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)
    if pattern != "random":
        # exact levels: the oracle's and the GPU's scores tie in the same groups
        assert len(np.unique(R)) == len(np.unique(s_np)) == (1 if pattern == "uniform" else 3)
        assert np.array_equal(g_sel, want), pattern
    else:
        band = check_selection(g_sel, R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks,
                               f"long history {N}")
        if band == 0:
            assert np.array_equal(g_sel, want)


def test_launch_count(kvm):
    """kvm_launch_count counts this library's kernels: one per Mean-K build and
    per view assembly; scoring is pass 1, combine, pass 2 and reduce, and the
    selection one kernel for short histories, six for long ones."""
    wl = MID
    for N, n_score in ((wl.n_blocks, 5), (20000, 10)):
        w = wl.with_(n_blocks=N, view_blocks=100)
        ctx = _ctx(kvm, w, max_positions=w.view_blocks * 32)
        q = torch.randn(w.n_layers, w.n_queries, w.n_q_heads, w.head_dim,
                        device="cuda").to(torch.bfloat16)
        index = torch.randn(ctx.index_shape(), device="cuda").to(torch.bfloat16)
        scores = torch.empty(N, device="cuda")
        sel = torch.empty(w.view_blocks, dtype=torch.int32, device="cuda")
        n0 = kvm.launch_count()
        ctx.score_select(q, w.n_queries, index, N, scores, sel)
        assert kvm.launch_count() - n0 == n_score, N
        ctx.sync()
    kp = torch.zeros(ctx.block_shape(2), dtype=torch.bfloat16, device="cuda")
    n0 = kvm.launch_count()
    ctx.build_index(kp, 0, 2, index)
    ids = torch.tensor([0, 1], dtype=torch.int32, device="cuda")   # blocks of kp
    ctx.assemble_view(ids, None, 2, kp, None, torch.empty_like(kp), None)
    assert kvm.launch_count() - n0 == 2
    ctx.sync()


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_assemble_view(kvm, wl):
    from paged_kv_cache_meank_gb300 import workload
    ws = workload.make_workspace(wl, seed=4, with_q=False)
    N, V = wl.n_blocks, wl.view_blocks
    ctx = _ctx(kvm, wl)
    rng = np.random.default_rng(5)
    ids = np.sort(rng.choice(N, size=V, replace=False)).astype(np.int32)
    pages = rng.permutation(V + 3)[:V].astype(np.int32)
    raw_d = ws.raw_k.to("cuda")
    v_d = ws.v.to("cuda")
    kp = torch.full(ctx.block_shape(V + 3), 3.0, dtype=ctx.kv_dtype, device="cuda")
    vp = torch.full(ctx.block_shape(V + 3), 3.0, dtype=ctx.kv_dtype, device="cuda")
    ctx.assemble_view(torch.from_numpy(ids).cuda(), torch.from_numpy(pages).cuda(), V, raw_d,
                      v_d, kp, vp)
    ctx.sync()
    raw = to_np(ws.raw_k, wl.kv_dtype)
    ref = ora.view_k(raw[ids], wl.kv_dtype, wl.rope_theta)
    got = to_np(kp, wl.kv_dtype)[pages]
    exact = assert_storage_close(got, ref, wl.kv_dtype, wl.name + " view K")
    assert exact > 0.999
    assert np.array_equal(to_np(vp, wl.kv_dtype)[pages], to_np(ws.v, wl.kv_dtype)[ids])
    untouched = sorted(set(range(V + 3)) - set(pages.tolist()))
    assert torch.all(kp[untouched].float() == 3.0) and torch.all(vp[untouched].float() == 3.0)
    # without page ids slot j lands in page j; without V only K is written
    kp2 = torch.zeros(ctx.block_shape(V), dtype=ctx.kv_dtype, device="cuda")
    ctx.assemble_view(torch.from_numpy(ids).cuda(), None, V, raw_d, None, kp2, None)
    ctx.sync()
    assert torch.equal(kp2, kp[torch.from_numpy(pages).long().cuda()])


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_assemble_roundtrip_at_original_positions(kvm, kv_dtype):
    """Every block selected in order lands at its original positions: the view
    K equals the prefill K (KVMem §4.4; InferScale Theorem 6)."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=40, view_blocks=40, kv_dtype=kv_dtype)
    ws = workload.make_workspace(wl, seed=6, with_q=False)
    raw = to_np(ws.raw_k, kv_dtype)
    kp_ref = prefill_k_pages(raw, kv_dtype, wl.rope_theta)
    ctx = _ctx(kvm, wl)
    out = torch.empty(ctx.block_shape(40), dtype=ctx.kv_dtype, device="cuda")
    ids = torch.arange(40, dtype=torch.int32, device="cuda")
    ctx.assemble_view(ids, None, 40, ws.raw_k.cuda(), None, out, None)
    ctx.sync()
    assert np.array_equal(to_np(out, kv_dtype), kp_ref)


def test_pinned_host_buffers(kvm):
    """Every call accepts pinned host buffers, which the kernels read over the
    host link; the results are bit-identical to the same calls on device
    buffers.  Pageable host memory and a host index on the device path are
    rejected."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=120, view_blocks=40)
    ws = workload.make_workspace(wl, seed=31)
    ctx = _ctx(kvm, wl)
    N, V = wl.n_blocks, wl.view_blocks
    kp = from_np(prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta), "bf16")

    def run(kp_in, v_in, q_in):
        index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
        raw = torch.empty(ctx.block_shape(N), dtype=torch.bfloat16, device="cuda")
        ctx.build_index(kp_in, 0, N, index, raw)
        scores = torch.empty(N, device="cuda")
        sel = torch.empty(V, dtype=torch.int32, device="cuda")
        ctx.score_select(q_in, wl.n_queries, index, N, scores, sel)
        k_out = torch.empty(ctx.block_shape(V), dtype=torch.bfloat16, device="cuda")
        v_out = torch.empty_like(k_out)
        ctx.assemble_view(sel, None, V, raw, v_in, k_out, v_out)
        ctx.sync()
        return index, raw, scores, sel, k_out, v_out

    dev = run(kp, ws.v.cuda(), ws.q.cuda())
    host = run(kp.cpu().pin_memory(), ws.v.pin_memory(), ws.q.pin_memory())
    for a, b in zip(dev, host):
        assert torch.equal(a, b)
    with pytest.raises(kvm.KvmError) as ei:                  # pageable memory
        ctx.build_index(kp.cpu(), 0, N, dev[0], None)
    assert ei.value.name == "KVM_ERR_INVALID_ARG"
    with pytest.raises(kvm.KvmError):                        # index on the TMA path
        ctx.score_select(ws.q.cuda(), wl.n_queries, dev[0].cpu().pin_memory(), N, dev[2],
                         dev[3])


def test_device_range_checks(kvm):
    """Out-of-range ids are skipped and reported by kvm_sync, and the context
    stays usable."""
    wl = MID64
    ctx = _ctx(kvm, wl)
    raw = torch.zeros(ctx.block_shape(4), dtype=torch.bfloat16, device="cuda")
    pages = torch.zeros(ctx.block_shape(4), dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([0, wl.n_blocks + 10], dtype=torch.int32, device="cuda")
    ctx.assemble_view(bad, None, 2, raw, None, pages, None)
    with pytest.raises(kvm.KvmError) as ei:
        ctx.sync()
    assert ei.value.name == "KVM_ERR_DEVICE"
    ok = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ctx.assemble_view(ok, None, 2, raw, None, pages, None)
    ctx.sync()


def test_host_side_errors(kvm):
    wl = MID64
    ctx = _ctx(kvm, wl)
    q = torch.zeros(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim, dtype=torch.bfloat16,
                    device="cuda")
    index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
    scores = torch.empty(wl.n_blocks + 10, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    with pytest.raises(kvm.KvmError) as ei:
        ctx.score_select(q, wl.n_queries, index, wl.n_blocks + 1, scores, sel)
    assert ei.value.name == "KVM_ERR_CAPACITY"
    with pytest.raises(kvm.KvmError) as ei:
        ctx.score_select(q, wl.n_queries + 1, index, wl.n_blocks, scores, sel)
    assert ei.value.name == "KVM_ERR_CAPACITY"
    with pytest.raises(kvm.KvmError) as ei:
        ctx.build_index(q, wl.n_blocks, 1, index)
    assert ei.value.name == "KVM_ERR_CAPACITY"
    with pytest.raises(kvm.KvmError) as ei:
        ctx.step(q, wl.n_queries, wl.n_blocks)
    assert ei.value.name == "KVM_ERR_NOT_BOUND"
    # still usable
    ctx.score_select(q, wl.n_queries, index, wl.n_blocks, scores, sel)
    ctx.sync()
