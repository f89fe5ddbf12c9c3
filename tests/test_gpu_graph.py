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
            st = eager.step(qs[i], wl.n_queries, wl.n_blocks)
            q_static.copy_(qs[i])
            g.replay()
            # the launch's counters equal the eager step's
            gst = graphed.graph_step_stats(s)
            eager.sync(s)
            assert dict(gst) == dict(st), f"step {t}: counters"
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
    on the host, scoring of a host-resident index and kvm_stage_out return
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
    blk = torch.zeros(host_diff.block_shape(1), dtype=torch.bfloat16, device="cuda")
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
        codes.append(host_diff.lib.kvm_stage_out(host_diff.handle, blk.data_ptr(),
                                                 blk.data_ptr(), 0, 1, cs))
        x.add_(1)
    g.replay()
    torch.cuda.synchronize()
    assert [STATUS[c] for c in codes] == ["KVM_ERR_INVALID_ARG"] * 4
    # no step of these contexts was captured: no graph counters to read
    for ctx in (dev, host_diff):
        with pytest.raises(kvm.KvmError) as ei:
            ctx.graph_step_stats(s)
        assert ei.value.name == "KVM_ERR_INVALID_ARG"
    assert x.tolist() == [1.0] * 4
    # the refused steps changed nothing: the first eager step misses every block
    with torch.cuda.stream(s):
        st = dev.step(q, wl.n_queries, wl.n_blocks)
        dev.sync(s)
    assert (st["hits"], st["misses"]) == (0, wl.view_blocks)


def test_graph_launch_waits_for_stage_out(kvm):
    """A step captured while the pinned host repository is still empty; the
    index is then built and the repository staged out chunk by chunk (262 MB
    of raw K and V on the copy stream), and the graph launched at once, with
    no sync.
    The launch waits for the stage-out copies through its external event
    wait, so its view equals an eager step's over the same repository."""
    from paged_kv_cache_meank_gb300 import workload
    from gpu_helpers import from_np, to_np
    from recall_ref import prefill_k_pages
    wl = MID.with_(n_blocks=2000, view_blocks=60)
    N, V = wl.n_blocks, wl.view_blocks
    ws = workload.make_workspace(wl, seed=67)
    kp = prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta)
    q = ws.q.cuda()
    s = torch.cuda.Stream()
    outs = []
    for graphed in (False, True):
        cfg = kvm.config_for(wl, repo_location=kvm.KVM_HOST_PINNED, h2d_mode=1)
        ctx = kvm.Context(cfg)
        raw_h = torch.zeros(ctx.block_shape(N), dtype=ctx.kv_dtype, pin_memory=True)
        v_h = torch.zeros_like(raw_h, pin_memory=True)
        index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
        P = cfg.pool_pages
        b = {"pool_k": torch.zeros(ctx.block_shape(P), dtype=ctx.kv_dtype, device="cuda")}
        b["pool_v"] = torch.zeros_like(b["pool_k"])
        b["pool_raw_k"] = torch.zeros_like(b["pool_k"])
        b["page_table"] = torch.empty(V, dtype=torch.int32, device="cuda")
        b["scores"] = torch.empty(N, device="cuda")
        b["sel_ids"] = torch.empty(V, dtype=torch.int32, device="cuda")
        ctx.bind(index=index, raw_k=raw_h, v=v_h, **b)
        torch.cuda.synchronize()
        if graphed:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                ctx.step(q, wl.n_queries, N)
        keep = []
        with torch.cuda.stream(s):
            for c0 in range(0, N, 256):
                n = min(256, N - c0)
                kp_d = from_np(kp[c0:c0 + n], "bf16")
                v_d = ws.v[c0:c0 + n].cuda()
                raw_d = torch.empty_like(kp_d)
                ctx.build_index(kp_d, c0, n, index, raw_d)
                ctx.stage_out(raw_d, v_d, c0, n)
                keep += [kp_d, v_d, raw_d]       # alive until the copies are done
            if graphed:
                g.replay()
            else:
                ctx.step(q, wl.n_queries, N)
            ctx.sync(s)
        outs.append(b)
    for k in _OUT + ("pool_raw_k",):
        assert torch.equal(outs[0][k], outs[1][k]), k
    pages = outs[1]["page_table"].long()
    sel = outs[1]["sel_ids"].long().cpu()
    assert torch.equal(outs[1]["pool_v"][pages].cpu(), ws.v[sel])


def test_build_score_assemble_capture(kvm):
    """kvm_build_index, kvm_score_select on a device index and
    kvm_assemble_view enqueue kernels on the caller's stream only: captured
    together into one graph, a launch gives the eager calls' index, raw K,
    scores, selection and view, bit for bit."""
    from paged_kv_cache_meank_gb300 import workload
    from gpu_helpers import from_np, to_np
    from recall_ref import prefill_k_pages
    wl = MID
    N, V = wl.n_blocks, wl.view_blocks
    ws = workload.make_workspace(wl, seed=69)
    kp = from_np(prefill_k_pages(to_np(ws.raw_k, "bf16"), "bf16", wl.rope_theta), "bf16")
    q, v = ws.q.cuda(), ws.v.cuda()
    ctx = kvm.Context(kvm.config_for(wl))
    s = torch.cuda.Stream()

    def buffers():
        return {"index": torch.zeros(ctx.index_shape(), dtype=ctx.index_dtype, device="cuda"),
                "raw": torch.empty(ctx.block_shape(N), dtype=ctx.kv_dtype, device="cuda"),
                "scores": torch.empty(N, device="cuda"),
                "sel": torch.empty(V, dtype=torch.int32, device="cuda"),
                "k": torch.empty(ctx.block_shape(V), dtype=ctx.kv_dtype, device="cuda"),
                "v": torch.empty(ctx.block_shape(V), dtype=ctx.kv_dtype, device="cuda")}

    def calls(b):
        ctx.build_index(kp, 0, N, b["index"], b["raw"])
        ctx.score_select(q, wl.n_queries, b["index"], N, b["scores"], b["sel"])
        ctx.assemble_view(b["sel"], None, V, b["raw"], v, b["k"], b["v"])

    eager, graphed = buffers(), buffers()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        calls(eager)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls(graphed)
    with torch.cuda.stream(s):
        g.replay()
        ctx.sync(s)
    for k in eager:
        assert torch.equal(eager[k], graphed[k]), k
