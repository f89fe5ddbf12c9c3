"""kvm_step captured into a CUDA graph, through the C ABI: each launch of the
graph runs one working-set step (the delta working set of KVMem §4.4) on the
query buffer as it holds at launch time, and gives the same scores,
selection, page table and pages as the same steps enqueued eagerly on a twin
context, including after a pool reset issued between launches.  Steps that
cannot be captured are refused before anything is enqueued."""
import pytest
import torch

from gpu_helpers import MID
from test_gpu_residency import _context, _queries

pytestmark = pytest.mark.gpu

_OUT = ("scores", "sel_ids", "page_table", "pool_k", "pool_v")


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    return kvm


@pytest.mark.parametrize("variant,repo_host,cfg_kw", [
    (0, False, {}),
    (0, True, {"delta_rerope_limit": 2}),
    (0, False, {"candidate_mode": 1}),
    (2, False, {}),
], ids=["two-pass-repo-device", "two-pass-repo-host-pull-delta", "two-pass-candidates",
        "one-launch-repo-device"])
def test_graph_launches_match_eager_steps(kvm, variant, repo_host, cfg_kw):
    """Six launches of one captured step, the queries changed in place
    between them, against six eager steps on a twin context; both pools are
    reset after the fourth step."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=400, view_blocks=48)
    ws = workload.make_workspace(wl, seed=61)
    qs = _queries(wl, 3, 62)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eager, be = _context(kvm, wl, ws, repo_host, 1, 0, score_variant=variant, **cfg_kw)
        graphed, bg = _context(kvm, wl, ws, repo_host, 1, 0, score_variant=variant, **cfg_kw)
    q_static = qs[0].clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert graphed.step(q_static, wl.n_queries, wl.n_blocks) is None
    with torch.cuda.stream(s):
        for t, i in enumerate([0, 1, 1, 2, 0, 2]):
            eager.step(qs[i], wl.n_queries, wl.n_blocks)
            q_static.copy_(qs[i])
            g.replay()
            if t == 3:
                eager.reset_pool()
                graphed.reset_pool()
            s.synchronize()
            for k in _OUT:
                assert torch.equal(be[k], bg[k]), f"step {t}: {k}"
        eager.sync(s)
        graphed.sync(s)


def test_eager_steps_and_graph_launches_interleave(kvm):
    """Eager steps and graph launches on one context share its residency: a
    launch after an eager step on the same queries finds every block resident,
    and the eager counters stay right around the launches."""
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(n_blocks=300, view_blocks=40)
    ws = workload.make_workspace(wl, seed=63)
    q0, q1 = _queries(wl, 2, 64)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ctx, b = _context(kvm, wl, ws, False, 1, 0)
        twin, bt = _context(kvm, wl, ws, False, 1, 0)
    q_static = q1.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ctx.step(q_static, wl.n_queries, wl.n_blocks)
    with torch.cuda.stream(s):
        st0 = ctx.step(q0, wl.n_queries, wl.n_blocks)
        g.replay()                                   # q1
        st1 = ctx.step(q1, wl.n_queries, wl.n_blocks)
        g.replay()                                   # q1 again
        st2 = ctx.step(q0, wl.n_queries, wl.n_blocks)
        for q in (q0, q1, q1, q1, q0):
            twin.step(q, wl.n_queries, wl.n_blocks)
        ctx.sync(s)
        twin.sync(s)
    assert (st0["hits"], st0["misses"]) == (0, wl.view_blocks)
    assert (st1["hits"], st1["misses"], st1["reroped"]) == (wl.view_blocks, 0, 0)
    for k in _OUT:
        assert torch.equal(b[k], bt[k]), k
    assert st2["hits"] + st2["misses"] == wl.view_blocks


def test_capture_refusals(kvm):
    """Under capture, kvm_step with a stats pointer, kvm_step whose diff runs
    on the host, and scoring of a host-resident index return
    KVM_ERR_INVALID_ARG and enqueue nothing; the capture itself stays valid."""
    import ctypes
    from paged_kv_cache_meank_gb300 import workload
    from paged_kv_cache_meank_gb300._abi import STATUS
    wl = MID.with_(n_blocks=200, view_blocks=40)
    ws = workload.make_workspace(wl, seed=65)
    q = _queries(wl, 1, 66)[0]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dev, _ = _context(kvm, wl, ws, False, 1, 0)
        host_diff, _ = _context(kvm, wl, ws, True, 0, 0)     # copy-engine transfers
        host_idx = kvm.Context(kvm.config_for(wl, index_location=kvm.KVM_HOST_PINNED))
    index_h = torch.zeros(host_idx.index_shape(), dtype=host_idx.index_dtype).pin_memory()
    scores = torch.empty(wl.n_blocks, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    x = torch.zeros(4, device="cuda")
    codes = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cs = s.cuda_stream
        st = kvm.KvmStepStats()
        codes.append(dev.lib.kvm_step(dev.handle, q.data_ptr(), wl.n_queries, wl.n_blocks,
                                      ctypes.byref(st), cs))
        codes.append(host_diff.lib.kvm_step(host_diff.handle, q.data_ptr(), wl.n_queries,
                                            wl.n_blocks, None, cs))
        codes.append(host_idx.lib.kvm_score_select(host_idx.handle, q.data_ptr(), wl.n_queries,
                                                   index_h.data_ptr(), wl.n_blocks,
                                                   scores.data_ptr(), sel.data_ptr(), None, cs))
        x.add_(1)
    g.replay()
    torch.cuda.synchronize()
    assert [STATUS[c] for c in codes] == ["KVM_ERR_INVALID_ARG"] * 3
    assert x.tolist() == [1.0] * 4
    # the refused steps changed nothing: the first eager step misses every block
    with torch.cuda.stream(s):
        st = dev.step(q, wl.n_queries, wl.n_blocks)
        dev.sync(s)
    assert (st["hits"], st["misses"]) == (0, wl.view_blocks)
