"""The oracle end to end on the tiny correctness workspace (no GPU)."""
import numpy as np

import oracle.kvmem as ora
from paged_kv_cache_meank_gb300 import configs, workload
from recall_ref import prefill_k_pages, recall, to_np


def test_tiny_workspace_recall():
    wl = configs.TINY
    ws = workload.make_workspace(wl, seed=0)
    raw = to_np(ws.raw_k, wl.kv_dtype)
    kp = prefill_k_pages(raw, wl.kv_dtype, wl.rope_theta)
    out = recall(wl, kp, to_np(ws.v, wl.kv_dtype), to_np(ws.q, wl.q_dtype))
    R, sel = out["R"], out["sel"]
    assert abs(R.sum() - wl.n_queries) < 1e-10
    assert len(sel) == wl.view_blocks == 13
    assert np.all(np.diff(sel) > 0)
    assert 0 in sel and all(b in sel for b in range(124, 128))
    # the six planted needles carry the query direction: all of them rank into the top-8
    planted = ws.planted.tolist()
    assert len(planted) == 6
    assert set(planted) <= set(sel.tolist()), (planted, sel)
    # Mean-K of the un-rotated prefill K is the mean of the raw K that made it
    mean_raw = raw.mean(axis=3).transpose(1, 2, 0, 3)
    assert np.max(np.abs(out["index"] - mean_raw)) < 1e-5
    # V bytes are copied unchanged
    assert np.array_equal(out["view_v"], to_np(ws.v, wl.kv_dtype)[sel])
    pos = ora.slot_positions(len(sel))
    assert pos.min() == 0 and pos.max() == 415


def test_history_shorter_than_reserved_blocks():
    """A history shorter than sink + recent has no candidate block to plant:
    the generator returns no planted ids and still draws K, V and queries."""
    wl = configs.TINY.with_(n_blocks=3, sink_blocks=1, recent_blocks=4, view_blocks=13)
    ws = workload.make_workspace(wl, seed=0)
    assert ws.planted.numel() == 0
    assert tuple(ws.raw_k.shape) == (3, wl.n_layers, wl.n_kv_heads, 32, wl.head_dim)
    assert ws.q.shape[1] == wl.n_queries
    ws2 = workload.make_index_direct(wl.with_(n_blocks=5), seed=0)
    assert ws2.planted.numel() == 0
