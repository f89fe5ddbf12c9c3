"""The kvm_step harness shared by the step tests: builds a context over a seeded
workspace (the GPU builds the index and raw K from the oracle's prefill K
pages), runs consecutive steps and checks each against the oracle: scores,
selection (band rule), the delta working set applied to the GPU's selection,
hit / miss / re-RoPE / H2D counts and the materialised view."""
import numpy as np
import torch

import oracle.kvmem as ora
import oracle.tier as oracle_tier
from gpu_helpers import (assert_meank_close, assert_scores_close, assert_storage_close,
                         check_selection, from_np, to_np)
from recall_ref import prefill_k_pages


def run_steps(kvm, wl, repo_host: bool, index_host: bool, queries, n_blocks_per_step,
               pool_extra=6, batch=7, h2d_mode=0, host_tier=None, index_spill=0,
               spill_tiles=0):
    from paged_kv_cache_meank_gb300 import workload
    N_max = max(n_blocks_per_step)
    ws = workload.make_workspace(wl, seed=11, n_blocks=N_max, with_q=False)
    raw_np = to_np(ws.raw_k, wl.kv_dtype)
    v_np = to_np(ws.v, wl.kv_dtype)
    kp = prefill_k_pages(raw_np, wl.kv_dtype, wl.rope_theta)
    cfg = kvm.config_for(
        wl, max_blocks=N_max, pool_pages=wl.view_blocks + pool_extra,
        repo_location=kvm.KVM_HOST_PINNED if repo_host else kvm.KVM_DEVICE,
        index_location=kvm.KVM_HOST_PINNED if index_host else kvm.KVM_DEVICE,
        h2d_batch_blocks=batch, h2d_mode=h2d_mode,
        host_tier_blocks=host_tier[0] if host_tier else 0,
        host_tier_lambda=host_tier[1] if host_tier else 0.5, index_spill=index_spill,
        spill_tiles=spill_tiles)
    cfg.tile_blocks = 64
    tier_ref = oracle_tier.HostTier(*host_tier) if host_tier else None
    ctx = kvm.Context(cfg)
    # (a) the GPU builds the index and raw K from the prefill K pages
    index_d = torch.zeros(ctx.index_shape(), dtype=ctx.index_dtype, device="cuda")
    raw_d = torch.empty(ctx.block_shape(N_max), dtype=ctx.kv_dtype, device="cuda")
    ctx.build_index(from_np(kp, wl.kv_dtype), 0, N_max, index_d, raw_d)
    ctx.sync()
    v_d = from_np(v_np, wl.kv_dtype)
    if repo_host:
        raw_repo = torch.empty(raw_d.shape, dtype=raw_d.dtype, pin_memory=True)
        raw_repo.copy_(raw_d)
        v_repo = torch.empty(v_d.shape, dtype=v_d.dtype, pin_memory=True)
        v_repo.copy_(v_d)
    else:
        raw_repo, v_repo = raw_d, v_d
    if index_host:
        index = torch.empty(index_d.shape, dtype=index_d.dtype, pin_memory=True)
        index.copy_(index_d)
    else:
        index = index_d
    P = cfg.pool_pages
    pool_k = torch.zeros(ctx.block_shape(P), dtype=ctx.kv_dtype, device="cuda")
    pool_v = torch.zeros_like(pool_k)
    pool_raw = torch.zeros_like(pool_k) if repo_host else None
    page_table = torch.full((wl.view_blocks,), -1, dtype=torch.int32, device="cuda")
    scores = torch.empty(N_max, device="cuda")
    sel = torch.empty(wl.view_blocks, dtype=torch.int32, device="cuda")
    ctx.bind(index=index, raw_k=raw_repo, v=v_repo, pool_k=pool_k, pool_v=pool_v,
             pool_raw_k=pool_raw, page_table=page_table, scores=scores, sel_ids=sel)

    # the oracle's own chain: Mean-K and raw K from the same prefill pages
    index_ref = ora.meank(kp, wl.kv_dtype, 0, wl.rope_theta)
    raw_ref = ora.raw_k(kp, wl.kv_dtype, 0, wl.rope_theta)
    rms = float(np.sqrt(np.mean(ora.as_f64(raw_np, wl.kv_dtype) ** 2)))
    kmax = float(np.abs(ora.as_f64(kp, wl.kv_dtype)).max()) * 2 ** 0.5
    assert_meank_close(to_np(index_d[:, :, :N_max], wl.index_dtype), index_ref,
                       wl.index_dtype, rms, "index", kmax)
    index_ref_stored = ora.as_f64(ora.round_to(index_ref.astype(np.float32), wl.index_dtype),
                                  wl.index_dtype)
    bop, bp = [-1] * P, [-1] * P
    history = []
    for step, (q, N) in enumerate(zip(queries, n_blocks_per_step)):
        st = ctx.step(q.to("cuda"), wl.n_queries, N)
        ctx.sync()
        R = ora.block_relevance(ora.as_f64(to_np(q, wl.q_dtype), wl.q_dtype),
                                index_ref_stored, N)
        assert_scores_close(scores[:N].cpu().numpy(), R, f"step {step}")
        g_sel = sel[:min(N, wl.view_blocks)].cpu().numpy()
        check_selection(g_sel, R, wl.sink_blocks, wl.recent_blocks, wl.view_blocks,
                        f"step {step}")
        # residency: the oracle's delta rule applied to the GPU's selection
        page, hit, rope, bop, bp = ora.residency_step(bop, bp, g_sel)
        assert page_table[:len(g_sel)].cpu().tolist() == page, f"step {step} page table"
        assert st["hits"] == sum(hit) and st["misses"] == len(hit) - sum(hit)
        assert st["reroped"] == sum(rope)
        if tier_ref is not None:   # the host-tier policy fed with this step's selection
            h, m, dem = tier_ref.step(g_sel.tolist(), N)
            assert (st["host_hits"], st["host_misses"], st["host_demoted"]) == (h, m, len(dem))
        blk = ctx.block_shape(1)
        nbytes = int(np.prod(blk)) * {"f32": 4, "bf16": 2, "e4m3": 1}[wl.kv_dtype]
        if repo_host:
            assert st["h2d_bytes"] == 2 * nbytes * st["misses"]
        # the view: K at compact positions from the oracle's raw K, V unchanged
        got_k = to_np(pool_k, wl.kv_dtype)[page]
        ref_k = ora.view_k(raw_ref[g_sel], wl.kv_dtype, wl.rope_theta)
        assert_storage_close(got_k, ref_k, wl.kv_dtype, f"step {step} view K")
        assert np.array_equal(to_np(pool_v, wl.kv_dtype)[page], v_np[g_sel])
        if repo_host:
            assert np.array_equal(to_np(pool_raw, wl.kv_dtype)[page], to_np(raw_d, wl.kv_dtype)[g_sel])
        history.append(st)
    return history
