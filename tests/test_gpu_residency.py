"""The residency diff of kvm_step on the device (the delta working set of
KVMem §4.4), through the C ABI: steps enqueued back to back with no wait on
the host give the pages and counters of the oracle's residency rule applied
to each step's selection, including more steps than the counter ring holds
between two syncs; the copy-engine path, whose diff runs on the host, gives
the same pages; a failed launch inside a step empties the pool and the next
step rebuilds it."""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import MID, assert_storage_close, from_np, to_np
from recall_ref import prefill_k_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return kvm


def _context(kvm, wl, ws, repo_host, h2d_mode, seed_q, **cfg_kw):
    """A bound context over the workspace, plus its pool and outputs."""
    N = wl.n_blocks
    cfg = kvm.config_for(wl, pool_pages=wl.view_blocks + 6,
                         repo_location=kvm.KVM_HOST_PINNED if repo_host else kvm.KVM_DEVICE,
                         h2d_mode=h2d_mode, **cfg_kw)
    ctx = kvm.Context(cfg)
    kp = prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta)
    index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
    raw = torch.empty(ctx.block_shape(N), dtype=torch.bfloat16, device="cuda")
    ctx.build_index(from_np(kp, "bf16"), 0, N, index, raw)
    ctx.sync()
    v = ws.v.cuda()
    if repo_host:
        raw, v = raw.cpu().pin_memory(), v.cpu().pin_memory()
    P = cfg.pool_pages
    bufs = {"pool_k": torch.zeros(ctx.block_shape(P), dtype=torch.bfloat16, device="cuda")}
    bufs["pool_v"] = torch.zeros_like(bufs["pool_k"])
    bufs["pool_raw_k"] = torch.zeros_like(bufs["pool_k"]) if repo_host else None
    bufs["page_table"] = torch.full((wl.view_blocks,), -1, dtype=torch.int32, device="cuda")
    bufs["scores"] = torch.empty(N, device="cuda")
    bufs["sel_ids"] = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.bind(index=index, raw_k=raw, v=v, **bufs)
    return ctx, bufs


def _queries(wl, n, seed):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim,
                        generator=g).to(torch.bfloat16).cuda() for _ in range(n)]


@pytest.mark.parametrize("repo_host", [False, True], ids=["repo-device", "repo-host-pull"])
def test_steps_back_to_back_match_the_residency_rule(kvm, repo_host):
    """Five steps are enqueued with no sync in between; each step's page table
    and counters equal the oracle's delta rule applied to that step's
    selection, and the page contents equal the host-diff (copy-engine) path's
    on the same selections."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=400, view_blocks=48)
    ws = workload.make_workspace(wl, seed=41)
    ctx, b = _context(kvm, wl, ws, repo_host, 1, 0)
    qs = _queries(wl, 3, 42)
    order = [0, 1, 1, 2, 0]                  # repeats give hits, moved hits and misses
    sels, pts, stats = [], [], []
    for i in order:
        stats.append(ctx.step(qs[i], wl.n_queries, wl.n_blocks))
        # copies of this step's outputs, on the same stream, before the next step
        sels.append(b["sel_ids"].clone())
        pts.append(b["page_table"].clone())
    ctx.sync()
    bop, bp = [-1] * ctx.cfg.pool_pages, [-1] * ctx.cfg.pool_pages
    for t, st in enumerate(stats):
        g_sel = sels[t].cpu().numpy()
        page, hit, rope, bop, bp = ora.residency_step(bop, bp, g_sel)
        assert pts[t].cpu().tolist() == page, f"step {t} page table"
        assert (st["hits"], st["misses"], st["reroped"]) == (sum(hit), len(hit) - sum(hit),
                                                             sum(rope)), f"step {t} counters"
        assert st["n_sel"] == wl.view_blocks and st["n_blocks"] == wl.n_blocks
    if repo_host:
        # the host-diff path (copy-engine transfers) on the same selections
        ctx2, b2 = _context(kvm, wl, ws, True, 0, 0)
        for i in order:
            ctx2.step(qs[i], wl.n_queries, wl.n_blocks)
            ctx2.sync()
        assert torch.equal(b2["page_table"], b["page_table"])
        pages = b["page_table"].long()
        assert torch.equal(b2["pool_k"][pages], b["pool_k"][pages])
        assert torch.equal(b2["pool_v"][pages], b["pool_v"][pages])


def test_more_steps_than_the_counter_ring(kvm):
    """70 steps between two syncs: the oldest counters are copied out when the
    64-slot ring is full, and every step's counters are right; steps without
    a stats pointer do not overwrite a waiting step's counters."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=200, view_blocks=40)
    ws = workload.make_workspace(wl, seed=43)
    ctx, b = _context(kvm, wl, ws, False, 1, 0)
    q = _queries(wl, 1, 44)[0]
    stats = [ctx.step(q, wl.n_queries, wl.n_blocks) for _ in range(70)]
    ctx.sync()
    assert stats[0]["misses"] == wl.view_blocks and stats[0]["hits"] == 0
    for st in stats[1:]:       # the same queries again: every block is a resident hit
        assert (st["hits"], st["misses"], st["reroped"]) == (wl.view_blocks, 0, 0)
    # a step with stats, then 70 steps without (a NULL stats pointer still
    # takes a ring slot): the first step's counters survive until the sync
    ctx.reset_pool()
    first = ctx.step(q, wl.n_queries, wl.n_blocks)
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(70):
        assert ctx.lib.kvm_step(ctx.handle, q.data_ptr(), wl.n_queries, wl.n_blocks, None, s) == 0
    ctx.sync()
    assert (first["misses"], first["hits"]) == (wl.view_blocks, 0)


def test_failed_launch_empties_the_pool(kvm):
    """An injected launch failure before the diff or before the assembly
    returns KVM_ERR_INJECTED; the pool is forgotten and the next step misses
    every block again and matches the oracle's view."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=200, view_blocks=40)
    ws = workload.make_workspace(wl, seed=45)
    ctx, b = _context(kvm, wl, ws, False, 1, 0)
    q = _queries(wl, 1, 46)[0]
    ctx.step(q, wl.n_queries, wl.n_blocks)
    ctx.sync()
    for nth in (1, 2):
        ctx.debug_inject(2, nth)
        with pytest.raises(kvm.KvmError) as ei:
            ctx.step(q, wl.n_queries, wl.n_blocks)
        assert ei.value.name == "KVM_ERR_INJECTED"
        ctx.sync()
        st = ctx.step(q, wl.n_queries, wl.n_blocks)
        ctx.sync()
        assert st["misses"] == wl.view_blocks and st["hits"] == 0
    g_sel = b["sel_ids"].cpu().numpy()
    raw_ref = ora.raw_k(prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta),
                        "bf16", 0, wl.rope_theta)
    pages = b["page_table"].cpu().numpy()
    got = to_np(b["pool_k"], "bf16")[pages]
    ref = ora.view_k(raw_ref[g_sel], "bf16", wl.rope_theta)
    assert_storage_close(got, ref, "bf16", "view after recovery")
    assert np.array_equal(to_np(b["pool_v"], "bf16")[pages], to_np(ws.v, "bf16")[g_sel])
