"""The whole recall path through kvm_step against the oracle: Mean-K build,
scoring and selection, the delta working set over a bounded page pool, and the
materialised view, over several consecutive steps, with the history's raw K / V
in device memory or in pinned host memory (packed, pipelined H2D)."""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import MID, assert_storage_close, from_np, to_np
from recall_ref import prefill_k_pages
from step_helpers import run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    return kvm


@pytest.mark.parametrize("repo_host,h2d_mode", [(False, 0), (True, 0), (True, 1)],
                         ids=["repo-device", "repo-host-copy-engine", "repo-host-gpu-pull"])
def test_step_sequence(kvm, repo_host, h2d_mode):
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    g = torch.Generator().manual_seed(21)
    u = workload.unit_vectors(2, wl.head_dim, g, "cpu")
    qa = workload.make_queries(wl, g, "cpu", u[0])
    qb = workload.make_queries(wl, g, "cpu", u[1])
    qs = [qa, qb, qb, qa]
    ns = [260, 280, 280, 300]   # the history grows between steps
    hist = run_steps(kvm, wl, repo_host, False, qs, ns, h2d_mode=h2d_mode)
    assert hist[0]["misses"] == wl.view_blocks and hist[0]["hits"] == 0
    # same queries, same history: every block is a hit and nothing moves
    assert hist[2]["misses"] == 0 and hist[2]["reroped"] == 0


@pytest.mark.parametrize("repo_host,h2d_mode", [(False, 0), (True, 1)],
                         ids=["repo-device", "repo-host-gpu-pull"])
def test_step_history_shrinks_and_grows(kvm, repo_host, h2d_mode):
    """The history shrinks between steps, below the view budget (50 blocks for
    60 slots: everything is selected, fewer slots than the budget), then grows
    back: pages holding blocks past the end are free, and blocks still resident
    from earlier steps are hits again."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    g = torch.Generator().manual_seed(23)
    u = workload.unit_vectors(2, wl.head_dim, g, "cpu")
    qa = workload.make_queries(wl, g, "cpu", u[0])
    qb = workload.make_queries(wl, g, "cpu", u[1])
    hist = run_steps(kvm, wl, repo_host, False, [qa, qb, qa, qa, qb], [300, 200, 50, 300, 300],
                      h2d_mode=h2d_mode)
    assert hist[2]["misses"] + hist[2]["hits"] == 50
    assert hist[3]["hits"] > 0 and hist[4]["hits"] > 0


@pytest.mark.parametrize("repo_host,h2d_mode", [(False, 0), (True, 0), (True, 1)],
                         ids=["repo-device", "repo-host-copy-engine", "repo-host-gpu-pull"])
def test_step_degenerate_histories(kvm, repo_host, h2d_mode):
    """Histories of 1 and 2 blocks (inside the sink window), exactly the view
    budget (60), one block more, and back to 1: the page table, counters and
    pages follow the oracle at every step, on the device-side diff (device
    repository, GPU pull) and the host-side one (copy engine)."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    g = torch.Generator().manual_seed(25)
    u = workload.unit_vectors(2, wl.head_dim, g, "cpu")
    qa = workload.make_queries(wl, g, "cpu", u[0])
    qb = workload.make_queries(wl, g, "cpu", u[1])
    hist = run_steps(kvm, wl, repo_host, False, [qa, qb, qa, qb, qa, qb],
                     [1, 2, 60, 61, 1, 60], h2d_mode=h2d_mode)
    assert [h["n_sel"] for h in hist] == [1, 2, 60, 60, 1, 60]
    assert hist[0]["misses"] == 1 and hist[1]["hits"] == 1 and hist[1]["misses"] == 1
    assert hist[4]["hits"] == 1 and hist[4]["misses"] == 0


@pytest.mark.parametrize("repo_host,h2d_mode", [(False, 0), (True, 0), (True, 1)],
                         ids=["repo-device", "repo-host-copy-engine", "repo-host-gpu-pull"])
def test_step_sequence_fp8_pages(kvm, repo_host, h2d_mode):
    """The same working-set sequence with 8-bit (e4m3) K / V pages: Mean-K from
    e4m3 prefill K, view K re-RoPE'd and rounded to e4m3, V bytes moved."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(kv_dtype="e4m3", name="mid-e4m3")
    g = torch.Generator().manual_seed(23)
    u = workload.unit_vectors(2, wl.head_dim, g, "cpu")
    qa = workload.make_queries(wl, g, "cpu", u[0])
    qb = workload.make_queries(wl, g, "cpu", u[1])
    hist = run_steps(kvm, wl, repo_host, False, [qa, qb, qa], [270, 290, 300],
                      h2d_mode=h2d_mode)
    assert hist[0]["misses"] == wl.view_blocks


def test_step_host_tier_policy(kvm):
    """kvm_step with host_tier_blocks: every step's selection feeds the LRFU
    host-tier policy; its hits, misses and demotions match the oracle's."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    g = torch.Generator().manual_seed(24)
    u = workload.unit_vectors(3, wl.head_dim, g, "cpu")
    qs = [workload.make_queries(wl, g, "cpu", u[k % 3]) for k in range(6)]
    hist = run_steps(kvm, wl, True, False, qs, [240, 250, 260, 270, 285, 300], h2d_mode=1,
                      host_tier=(wl.view_blocks + 20, 0.3))
    assert hist[0]["host_misses"] == 0          # all blocks are created resident
    assert sum(h["host_demoted"] for h in hist) > 0


@pytest.mark.parametrize("index_spill,spill_tiles", [(0, 0), (1, 0), (1, 2)],
                         ids=["restream", "spill", "spill-budget"])
def test_step_host_index_tiled(kvm, index_spill, spill_tiles):
    """Index in pinned host memory, scored in 64-block tiles (KVMem §5); with
    index_spill the tiles cross the host link once per step, or all but the
    last two of them twice under a two-tile budget."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID
    g = torch.Generator().manual_seed(22)
    u = workload.unit_vectors(1, wl.head_dim, g, "cpu")
    q = workload.make_queries(wl, g, "cpu", u[0])
    run_steps(kvm, wl, True, True, [q, q], [300, 300], index_spill=index_spill,
              spill_tiles=spill_tiles)


def test_step_failure_injection(kvm):
    """A failed copy submission or kernel launch inside kvm_step returns
    KVM_ERR_INJECTED; the pool is forgotten and the next step rebuilds it."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=200, view_blocks=40)
    ws = workload.make_workspace(wl, seed=13)
    ctx = kvm.Context(kvm.config_for(wl, repo_location=kvm.KVM_HOST_PINNED, h2d_batch_blocks=5,
                                     h2d_mode=0))       # copy-engine transfers can fail
    kp = prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta)
    index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
    ctx.build_index(from_np(kp, "bf16"), 0, 200, index, None)
    # the host repository holds the oracle's raw K of the same prefill pages
    raw_ref = ora.raw_k(kp, "bf16", 0, wl.rope_theta)
    raw_h = torch.empty(ctx.block_shape(200), dtype=torch.bfloat16, pin_memory=True)
    raw_h.copy_(from_np(raw_ref, "bf16"))
    v_h = ws.v.pin_memory()
    P = ctx.cfg.pool_pages
    pool_k = torch.zeros(ctx.block_shape(P), dtype=torch.bfloat16, device="cuda")
    pool_v, pool_r = torch.zeros_like(pool_k), torch.zeros_like(pool_k)
    pt = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    scores = torch.empty(200, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.bind(index=index, raw_k=raw_h, v=v_h, pool_k=pool_k, pool_v=pool_v, pool_raw_k=pool_r,
             page_table=pt, scores=scores, sel_ids=sel)
    q = ws.q.cuda()
    for what, nth in ((1, 3), (2, 2)):
        ctx.reset_pool()          # every selected block is a miss again
        ctx.debug_inject(what, nth)
        with pytest.raises(kvm.KvmError) as ei:
            ctx.step(q, wl.n_queries, 200)
        assert ei.value.name == "KVM_ERR_INJECTED"
        ctx.sync()
        st = ctx.step(q, wl.n_queries, 200)   # recovers: the pool starts empty again
        ctx.sync()
        assert st["misses"] == wl.view_blocks
    ref = ora.view_k(raw_ref[sel.cpu().numpy()], "bf16", wl.rope_theta)
    got = to_np(pool_k, "bf16")[pt.cpu().numpy()]
    assert_storage_close(got, ref, "bf16", "after recovery")


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("repo_host", [False, True], ids=["repo-device", "repo-host-pull-no-raw-copy"])
def test_step_bounded_delta_rerope(kvm, repo_host, dt):
    """Bounded delta re-RoPE (KVMem §4.4): hits whose slot moved are rotated in
    place by the position change at most once in a row, then rebuilt from raw K;
    every page is compared with the oracle's own pool that applies the same
    actions (delta rotation of its stored page, or RoPE of raw K).  Both page
    types: bf16, and e4m3 rotated in place from its 8-bit values."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(kv_dtype=dt)
    limit = 1
    N_max = 300
    ws = workload.make_workspace(wl, seed=61, n_blocks=N_max, with_q=False)
    raw_np, v_np = to_np(ws.raw_k, dt), to_np(ws.v, dt)
    kp = prefill_k_pages(raw_np, dt, wl.rope_theta)
    cfg = kvm.config_for(wl, max_blocks=N_max, pool_pages=wl.view_blocks + 6,
                         repo_location=kvm.KVM_HOST_PINNED if repo_host else kvm.KVM_DEVICE,
                         h2d_mode=1, delta_rerope_limit=limit)
    ctx = kvm.Context(cfg)
    index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
    ctx.build_index(from_np(kp, dt), 0, N_max, index, None)
    ctx.sync()
    # the repository holds the oracle's raw K of the same prefill pages
    raw_ref = ora.raw_k(kp, dt, 0, wl.rope_theta)
    raw_d = from_np(raw_ref, dt)
    v_d = from_np(v_np, dt)
    if repo_host:
        raw_repo = torch.empty(raw_d.shape, dtype=raw_d.dtype, pin_memory=True)
        raw_repo.copy_(raw_d)
        v_repo = torch.empty(v_d.shape, dtype=v_d.dtype, pin_memory=True)
        v_repo.copy_(v_d)
    else:
        raw_repo, v_repo = raw_d, v_d
    P = cfg.pool_pages
    pool_k = torch.zeros(ctx.block_shape(P), dtype=ctx.kv_dtype, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    pt = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    scores = torch.empty(N_max, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.bind(index=index, raw_k=raw_repo, v=v_repo, pool_k=pool_k, pool_v=pool_v,
             pool_raw_k=None, page_table=pt, scores=scores, sel_ids=sel)
    g = torch.Generator().manual_seed(62)
    u = workload.unit_vectors(3, wl.head_dim, g, "cpu")
    qs = [workload.make_queries(wl, g, "cpu", u[i % 3]) for i in range(6)]
    ns = [240, 250, 260, 270, 285, 300]     # the history grows: selections shift slots
    bop, bp, cnt = [-1] * P, [-1] * P, [0] * P
    ora_pool = {}
    n_delta = n_rebuild = 0
    for step, (q, N) in enumerate(zip(qs, ns)):
        st = ctx.step(q.cuda(), wl.n_queries, N)
        ctx.sync()
        g_sel = sel[:wl.view_blocks].cpu().numpy()
        prev_bp = list(bp)
        page, act, bop, bp, cnt = ora.residency_step_delta(bop, bp, cnt, g_sel, limit)
        assert pt.cpu().tolist() == page, f"step {step} page table"
        assert st["delta_reroped"] == act.count("delta"), (step, st, act.count("delta"))
        for j, (p, a) in enumerate(zip(page, act)):
            if a in ("miss", "rebuild"):
                c, s = ora.cos_sin_f32(ora.slot_positions(j + 1)[j], wl.head_dim, wl.rope_theta)
                ora_pool[p] = ora.round_to(ora.rope_f32(ora.as_f32(raw_ref[g_sel[j]], dt), c, s),
                                           dt)
            elif a == "delta":
                ora_pool[p] = ora.delta_rerope_k(ora_pool[p][None], dt, j * 32 - prev_bp[p],
                                                 wl.rope_theta)[0]
        n_delta += act.count("delta")
        n_rebuild += act.count("rebuild")
        got = to_np(pool_k, dt)
        for j, p in enumerate(page):
            assert_storage_close(got[p][None], ora_pool[p][None], dt, f"step {step} slot {j}")
        assert np.array_equal(to_np(pool_v, dt)[page], v_np[g_sel])
    assert n_delta > 0 and n_rebuild > 0      # both branches of the bound were taken
