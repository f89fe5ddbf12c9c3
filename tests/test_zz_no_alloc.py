"""kvm_score_select_static: block scoring and selection for callers that cannot
allocate device memory.

Such callers exist: a plugin running inside an inference engine whose memory
planner already owns every byte of the device, or a latency-critical caller
that cannot pay for cudaMalloc / cudaFree (which may synchronise the device).
The entry point keeps its scratch in a fixed array inside the library, so it
needs no context and no workspace.  Here its output is checked against the
workspace-based kvm_score_select, within the parity tolerance the other tests
use, on calls in a row with different shapes (so anything left in the
shared scratch by one call would show up in the next).  The third call has
enough blocks for the many-CTA selection, whose histograms live in the shared
scratch and must start at zero on every call.
"""
import ctypes

import pytest
import torch

from gpu_helpers import MID, REL_SCORE
from paged_kv_cache_meank_gb300 import configs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvm():
    import paged_kv_cache_meank_gb300 as kvm
    from paged_kv_cache_meank_gb300 import build
    build.build()
    return kvm


def _compare(kvm, wl, seed):
    from paged_kv_cache_meank_gb300 import workload
    ws = workload.make_index_direct(wl, seed=seed, device="cuda")
    cfg = kvm.config_for(wl, index_location=kvm.KVM_DEVICE, repo_location=kvm.KVM_DEVICE)
    N, V = wl.n_blocks, wl.view_blocks
    # the existing entry point, with a context and its workspace
    ctx = kvm.Context(cfg)
    s_ref = torch.empty(N, device="cuda")
    sel_ref = torch.full((V,), -1, dtype=torch.int32, device="cuda")
    n_ref = ctx.score_select(ws.q, wl.n_queries, ws.index, N, s_ref, sel_ref)
    ctx.sync()
    # the allocation-free entry point
    s = torch.full((N,), float("nan"), device="cuda")
    sel = torch.full((V,), -1, dtype=torch.int32, device="cuda")
    n = kvm.score_select_static(cfg, ws.q, wl.n_queries, ws.index, N, s, sel)
    torch.cuda.synchronize()
    assert n == n_ref == min(N, V)
    rel = ((s.double() - s_ref.double()).abs() / s_ref.double().abs()).max().item()
    assert rel <= REL_SCORE, rel
    if torch.equal(s, s_ref):
        assert torch.equal(sel, sel_ref)
    else:  # scores differ within tolerance: the selections must agree outside near-ties
        assert len(set(sel.tolist()) ^ set(sel_ref.tolist())) <= 4
    ctx.close()


def test_static_matches_workspace_entry_point_on_calls_in_a_row(kvm):
    _compare(kvm, MID, seed=41)                       # call 1: small, 4 layers x 2 heads
    _compare(kvm, configs.W256K, seed=42)             # call 2: 64 x 8 heads, 8192 blocks
    many = MID.with_(name="mid-bf16-20000", n_blocks=20000, view_blocks=600)
    _compare(kvm, many, seed=43)                      # call 3: many-CTA selection
    _compare(kvm, many, seed=44)                      # call 4: its histograms cleared again


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
