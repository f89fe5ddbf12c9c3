"""Chunked prefill with incremental indexing and proactive stage-out (KVMem
§4.4 and §5): each completed chunk's Mean-K is built while its K is on the GPU
and its raw K / V are staged out to the host repository on the copy stream;
a working-set update then materialises the view from that repository."""
import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import MID, assert_meank_close, assert_storage_close, check_selection, from_np, to_np
from recall_ref import prefill_k_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    return kvm


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("h2d_mode", [0, 1], ids=["copy-engine", "gpu-pull"])
def test_chunked_prefill_stage_out_then_step(kvm, h2d_mode, dt):
    from paged_kv_cache_meank_gb300 import workload
    wl = MID.with_(kv_dtype=dt)
    N, V = wl.n_blocks, wl.view_blocks
    ws = workload.make_workspace(wl, seed=51)
    raw_np, v_np = to_np(ws.raw_k, dt), to_np(ws.v, dt)
    kp = prefill_k_pages(raw_np, dt, wl.rope_theta)
    cfg = kvm.config_for(wl, repo_location=kvm.KVM_HOST_PINNED, h2d_mode=h2d_mode,
                         h2d_batch_blocks=16)
    ctx = kvm.Context(cfg)
    raw_h = torch.zeros(ctx.block_shape(N), dtype=ctx.kv_dtype, pin_memory=True)
    v_h = torch.zeros_like(raw_h, pin_memory=True)
    index = torch.zeros(ctx.index_shape(), dtype=torch.bfloat16, device="cuda")
    P = cfg.pool_pages
    pool_k = torch.zeros(ctx.block_shape(P), dtype=ctx.kv_dtype, device="cuda")
    pool_v, pool_r = torch.zeros_like(pool_k), torch.zeros_like(pool_k)
    pt = torch.empty(V, dtype=torch.int32, device="cuda")
    scores = torch.empty(N, device="cuda")
    sel = torch.empty(V, dtype=torch.int32, device="cuda")
    ctx.bind(index=index, raw_k=raw_h, v=v_h, pool_k=pool_k, pool_v=pool_v, pool_raw_k=pool_r,
             page_table=pt, scores=scores, sel_ids=sel)
    keep = []
    for c0 in range(0, N, 64):                     # prefill chunks of 64 blocks, ragged tail
        n = min(64, N - c0)
        kp_d = from_np(kp[c0:c0 + n], dt)
        v_d = from_np(v_np[c0:c0 + n], dt)
        raw_d = torch.empty_like(kp_d)
        ctx.build_index(kp_d, c0, n, index, raw_d)
        ctx.stage_out(raw_d, v_d, c0, n)
        keep += [kp_d, v_d, raw_d]                 # alive until the copies are done
    st = ctx.step(ws.q.cuda(), wl.n_queries, N)    # ordered after every stage-out
    ctx.sync()
    del keep
    raw_ref = ora.raw_k(kp, dt, 0, wl.rope_theta)
    assert_storage_close(to_np(raw_h, dt), raw_ref, dt, "staged raw K")
    assert np.array_equal(to_np(v_h, dt), v_np)
    index_ref = ora.meank(kp, dt, 0, wl.rope_theta)
    kmax = float(np.abs(ora.as_f64(kp, dt)).max()) * 2 ** 0.5
    assert_meank_close(to_np(index[:, :, :N], "bf16"), index_ref, "bf16", wl.k_std, "index", kmax)
    R = ora.block_relevance(ora.as_f64(to_np(ws.q, "bf16"), "bf16"),
                            ora.as_f64(ora.round_to(index_ref.astype(np.float32), "bf16"), "bf16"),
                            N)
    g_sel = sel.cpu().numpy()
    check_selection(g_sel, R, wl.sink_blocks, wl.recent_blocks, V, "after stage-out")
    assert st["misses"] == V
    page = pt.cpu().numpy()
    got = to_np(pool_k, dt)[page]
    assert_storage_close(got, ora.view_k(raw_ref[g_sel], dt, wl.rope_theta), dt, "view K")
    assert np.array_equal(to_np(pool_v, dt)[page], v_np[g_sel])


def test_stage_out_needs_host_repository(kvm):
    wl = MID
    ctx = kvm.Context(kvm.config_for(wl))                         # device repository
    x = torch.zeros(ctx.block_shape(1), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvm.KvmError) as ei:
        ctx.stage_out(x, x, 0, 1)
    assert ei.value.name == "KVM_ERR_NOT_BOUND"
