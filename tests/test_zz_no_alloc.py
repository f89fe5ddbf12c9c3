"""kvm_score_select_static: block scoring and selection for callers that cannot
allocate device memory.

Such callers exist: a plugin running inside an inference engine whose memory
planner already owns every byte of the device, or a latency-critical caller
that cannot pay for cudaMalloc / cudaFree (which may synchronise the device).
The entry point keeps its scratch in a fixed array inside the library, so it
needs no context and no workspace.

Each call here is checked two ways: bit for bit against the workspace-based
kvm_score_select on the same inputs (same kernels, same chunking), and against
the float64 oracle with the parity rules of the other tests (scores within
1e-4 relative, selection by the near-tie band rule).  The calls run in a row
with different shapes, so anything one call left in the shared scratch would
show up in the next; two of them have enough blocks for the many-CTA
selection, whose histograms live in the shared scratch and must start at zero
on every call.  After the calls, the device error word reads clear.

This file is collected last, so that a run stopping at its first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.kvmem as ora
from gpu_helpers import MID, assert_scores_close, check_selection, to_np
from paged_kv_cache_meank_gb300 import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    return kvm


def _oracle_scores(wl, ws, candidate_mode):
    q = ora.as_f64(to_np(ws.q, wl.q_dtype), wl.q_dtype)
    idx = ora.as_f64(to_np(ws.index, wl.index_dtype), wl.index_dtype)
    if candidate_mode == 1:
        return ora.block_relevance_excl(q, idx, wl.n_blocks, wl.sink_blocks, wl.recent_blocks)
    return ora.block_relevance(q, idx, wl.n_blocks)


def _call_both(kvm, wl, seed, candidate_mode=0, oracle=True):
    """One static call and one workspace call on the same inputs; the static
    outputs must equal the workspace outputs bit for bit, and (with
    ``oracle``) match the oracle under the parity rules."""
    from paged_kv_cache_meank_gb300 import workload
    ws = workload.make_index_direct(wl, seed=seed, device="cuda")
    cfg = kvm.config_for(wl, max_blocks=wl.n_blocks, index_location=kvm.KVM_DEVICE,
                         repo_location=kvm.KVM_DEVICE, candidate_mode=candidate_mode)
    N, V = wl.n_blocks, wl.view_blocks
    ctx = kvm.Context(cfg)
    s_ref = torch.empty(N, device="cuda")
    sel_ref = torch.full((V,), -1, dtype=torch.int32, device="cuda")
    n_ref = ctx.score_select(ws.q, wl.n_queries, ws.index, N, s_ref, sel_ref)
    ctx.sync()
    s = torch.full((N,), float("nan"), device="cuda")
    sel = torch.full((V,), -1, dtype=torch.int32, device="cuda")
    n = kvm.score_select_static(cfg, ws.q, wl.n_queries, ws.index, N, s, sel)
    torch.cuda.synchronize()
    ctx.close()
    n_sel = min(N, V)
    assert n == n_ref == n_sel
    assert torch.equal(s, s_ref), (wl.name, "scores differ from kvm_score_select")
    assert torch.equal(sel, sel_ref), (wl.name, "selection differs from kvm_score_select")
    if oracle:
        R = _oracle_scores(wl, ws, candidate_mode)
        g = s.cpu().numpy()
        if candidate_mode == 1:
            c0, c1 = ora.candidate_range(N, wl.sink_blocks, wl.recent_blocks)
            assert np.all(g[:c0] == 0) and np.all(g[c1:] == 0)
            assert_scores_close(g[c0:c1], R[c0:c1], wl.name)
        else:
            assert_scores_close(g, R, wl.name)
        check_selection(sel[:n_sel].cpu().numpy(), R, wl.sink_blocks, wl.recent_blocks, V,
                        wl.name)


def test_static_matches_workspace_entry_point_and_oracle_on_calls_in_a_row(kvm):
    many = MID.with_(name="mid-bf16-20000", n_blocks=20000, view_blocks=600)
    _call_both(kvm, MID, seed=41)                                  # 4 layers x 2 kv heads
    _call_both(kvm, configs.W256K.with_(name="q27-256k-8l", n_layers=8), seed=42)
    _call_both(kvm, configs.W256K, seed=43, oracle=False)          # 16.8 MB of the scratch
    _call_both(kvm, many, seed=44)                                 # many-CTA selection
    _call_both(kvm, many, seed=45)                                 # its histograms cleared again
    _call_both(kvm, MID, seed=46, candidate_mode=1)                # reserved blocks left out
    kvm.score_select_static_status()                               # no device flag raised


def test_static_rejects_sizes_beyond_its_scratch(kvm):
    wl = configs.W10M                                  # 64 x 8 x 312500 blocks: ~640 MB
    cfg = kvm.config_for(wl, index_location=kvm.KVM_DEVICE, repo_location=kvm.KVM_DEVICE)
    lib = kvm.load()
    n_sel = ctypes.c_int32()
    dummy = ctypes.c_void_p(256)                       # never dereferenced: rejected first
    st = lib.kvm_score_select_static(ctypes.byref(cfg), dummy, wl.n_queries, dummy,
                                     wl.n_blocks, dummy, dummy, ctypes.byref(n_sel), None)
    assert st == -3                                    # KVM_ERR_CAPACITY
    assert b"scratch" in lib.kvm_last_error()


def test_static_rejects_buffers_the_kernels_cannot_use(kvm):
    """The index must be device memory; q and the outputs device or pinned
    host memory.  Pageable host buffers are rejected before anything runs."""
    wl = MID
    cfg = kvm.config_for(wl, max_blocks=wl.n_blocks, index_location=kvm.KVM_DEVICE,
                         repo_location=kvm.KVM_DEVICE)
    lib = kvm.load()
    n_sel = ctypes.c_int32()
    dev_q = torch.zeros(wl.n_layers, wl.n_queries, wl.n_q_heads, wl.head_dim,
                        dtype=torch.bfloat16, device="cuda")
    dev_idx = torch.zeros(wl.n_layers, wl.n_kv_heads, wl.n_blocks, wl.head_dim,
                          dtype=torch.bfloat16, device="cuda")
    dev_s = torch.zeros(wl.n_blocks, device="cuda")
    dev_sel = torch.zeros(wl.view_blocks, dtype=torch.int32, device="cuda")
    host_idx = dev_idx.cpu()                           # pageable
    host_s = torch.zeros(wl.n_blocks)                  # pageable

    def call(q, idx, s, sel):
        return lib.kvm_score_select_static(ctypes.byref(cfg), q.data_ptr(), wl.n_queries,
                                           idx.data_ptr(), wl.n_blocks, s.data_ptr(),
                                           sel.data_ptr(), ctypes.byref(n_sel), None)

    assert call(dev_q, host_idx, dev_s, dev_sel) == -1     # KVM_ERR_INVALID_ARG
    assert b"index" in lib.kvm_last_error()
    assert call(dev_q, dev_idx, host_s, dev_sel) == -1
    assert b"scores_out" in lib.kvm_last_error()
    assert call(dev_q.cpu(), dev_idx, dev_s, dev_sel) == -1
    assert b"q" in lib.kvm_last_error()
