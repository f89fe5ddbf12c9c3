"""Parity of the one-launch scoring variant (score_variant 2) against the CPU
oracle, through the C ABI.

Both softmax passes of Eq. (10) (KVMem §4.3) run in one persistent launch in
which groups of CTAs share a (layer, kv head) slice and fold their per-row
statistics across CTAs before pass 2.  The cases cover one and two pass-1 row
tiles (rows <= 128 and 129..192), shares that end on a half tile, candidate
sets with and without the reserved blocks, several slices per group, queries
in pinned host memory, the allocation-free entry point and the bounded waits.
"""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import MID, MID64, assert_scores_close, check_selection, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return kvm


def _oracle(ws, wl, N, candidate_mode=0):
    q = ora.as_f64(to_np(ws.q, "bf16"), "bf16")
    idx = ora.as_f64(to_np(ws.index, "bf16"), "bf16")
    if candidate_mode:
        return ora.block_relevance_excl(q, idx, N, wl.sink_blocks, wl.recent_blocks)
    return ora.block_relevance(q, idx, N)


def _run(kvm, wl, ws, N, q=None, **kw):
    ctx = kvm.Context(kvm.config_for(wl, score_variant=2, **kw))
    scores = torch.empty(N, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.score_select(ws.q.cuda() if q is None else q, wl.n_queries, ws.index.cuda(), N, scores,
                     sel)
    ctx.sync()
    return scores, sel


@pytest.mark.parametrize("n_queries,N", [(21, 517), (22, 517), (27, 3000), (32, 3000),
                                         (32, 4863), (16, 129)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("candidate_mode", [0, 1], ids=["all", "excl"])
def test_one_launch_parity(kvm, n_queries, N, candidate_mode):
    """126, 132, 162 and 192 query rows per KV head (one row tile; two row
    tiles overlapping at row 64 or 32), 96 rows, short and long histories."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=N, view_blocks=min(60, N), n_queries=n_queries)
    ws = workload.make_index_direct(wl, seed=70 + n_queries + N)
    scores, sel = _run(kvm, wl, ws, N, candidate_mode=candidate_mode)
    R = _oracle(ws, wl, N, candidate_mode)
    got = scores.cpu().numpy()
    if candidate_mode:
        S, W = wl.sink_blocks, wl.recent_blocks
        assert np.all(got[:S] == 0) and np.all(got[N - W:] == 0)
        assert_scores_close(got[S:N - W], R[S:N - W], "one launch, candidates only")
    else:
        assert_scores_close(got, R, "one launch")
        assert abs(got.sum() - wl.n_queries) < 1e-3 * wl.n_queries
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks,
                    "one launch")


def test_one_launch_d64_and_many_slices(kvm):
    """d = 64 (one K atom) with 12 (layer, kv head) slices, and d = 128 with 64
    slices over a history long enough for several CTAs per slice."""
    from paged_kv_cache_meank_gb300 import workload
    for wl in (MID64.with_(n_blocks=2049), MID.with_(n_layers=8, n_kv_heads=8, n_q_heads=48,
                                                     n_blocks=6001)):
        ws = workload.make_index_direct(wl, seed=91)
        scores, sel = _run(kvm, wl, ws, wl.n_blocks)
        R = _oracle(ws, wl, wl.n_blocks)
        assert_scores_close(scores.cpu().numpy(), R, wl.name)
        check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks,
                        wl.name)


def test_one_launch_host_queries_and_static_entry_point(kvm):
    """Queries in pinned host memory are copied to the workspace and take the
    same launch: bit-identical results.  The allocation-free entry point with
    score_variant 2 and device queries also matches bit for bit."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=1500)
    N = wl.n_blocks
    ws = workload.make_index_direct(wl, seed=92)
    dev = _run(kvm, wl, ws, N)
    host = _run(kvm, wl, ws, N, q=ws.q.pin_memory())
    assert torch.equal(dev[0], host[0]) and torch.equal(dev[1], host[1])
    cfg = kvm.config_for(wl, score_variant=2)
    scores = torch.empty(N, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    kvm.score_select_static(cfg, ws.q.cuda(), wl.n_queries, ws.index.cuda(), N, scores, sel)
    torch.cuda.synchronize()
    kvm.score_select_static_status()
    assert torch.equal(scores, dev[0]) and torch.equal(sel, dev[1])


@pytest.mark.parametrize("nth", [1, 2], ids=["pass1", "pass2"])
def test_one_launch_bounded_wait_and_recovery(kvm, nth):
    """The TMA producer skips pass 1 (or pass 2): the bounded waits run out,
    the group counters stop no CTA for long, kvm_sync reports KVM_ERR_TIMEOUT
    and the next call on the same context matches the oracle."""
    import time
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=2000)
    N = wl.n_blocks
    ws = workload.make_index_direct(wl, seed=93)
    ctx = kvm.Context(kvm.config_for(wl, score_variant=2))
    q, index = ws.q.cuda(), ws.index.cuda()
    scores = torch.empty(N, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.debug_inject(3, nth)
    t0 = time.monotonic()
    ctx.score_select(q, wl.n_queries, index, N, scores, sel)
    with pytest.raises(kvm.KvmError) as ei:
        ctx.sync()
    assert ei.value.name == "KVM_ERR_TIMEOUT"
    assert time.monotonic() - t0 < 30.0
    s = sel.cpu().numpy()
    assert np.all((s >= 0) & (s < N))
    ctx.score_select(q, wl.n_queries, index, N, scores, sel)
    ctx.sync()
    R = _oracle(ws, wl, N)
    assert_scores_close(scores.cpu().numpy(), R, "after a timed-out one-launch call")
    check_selection(sel.cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks)
