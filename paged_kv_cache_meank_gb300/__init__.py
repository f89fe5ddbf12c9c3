"""GB300-native per-step working-set recall for virtualised agent-workspace KV.

Thin Python binding over libkvm.so (include/kvm.h).  PyTorch provides device
memory, pinned host memory and streams; every step of the recall path runs in
the library's CUDA kernels.  The names follow the C ABI:

  Context.build_index    kvm_build_index    Mean-K index build
  Context.score_select   kvm_score_select   Eq. (10) scoring + budgeted top-k
  Context.assemble_view  kvm_assemble_view  gather + re-RoPE + V copy
  Context.step           kvm_step           one working-set update with page reuse

Sources: "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU"
(§4.3, §4.4, §5) and "InferScale: GPU-Native KV Injection for Personalized LLM
Serving" (§2 RoPE background, Theorem 6).
"""
from __future__ import annotations

import ctypes
from collections.abc import Mapping

import torch

from . import _abi
from ._abi import (KVM_BF16, KVM_DEVICE, KVM_E4M3, KVM_F32, KVM_HOST_PINNED, KvmBuffers,
                   KvmConfig, KvmError, KvmStepStats, KvmTierStats, check, load)
from .configs import BLOCK_TOKENS, Workload

__all__ = ["Context", "HostTier", "KvmError", "config_for", "launch_count", "load", "KVM_F32",
           "KVM_BF16", "KVM_E4M3", "KVM_DEVICE", "KVM_HOST_PINNED"]

_DT = {"f32": KVM_F32, "bf16": KVM_BF16, "e4m3": KVM_E4M3}
# e4m3 elements travel as their bit patterns in uint8 tensors
_TDT = {KVM_F32: torch.float32, KVM_BF16: torch.bfloat16, KVM_E4M3: torch.uint8}


def config_for(wl: Workload, *, max_blocks: int | None = None, max_positions: int | None = None,
               pool_pages: int | None = None, index_location: int | None = None,
               repo_location: int | None = None, h2d_batch_blocks: int = 64,
               max_queries: int | None = None, score_variant: int = 0,
               h2d_mode: int = 1, delta_rerope_limit: int = 0,
               candidate_mode: int = 0, host_tier_blocks: int = 0,
               host_tier_lambda: float = 0.5, index_spill: int = 0,
               spill_tiles: int = 0) -> KvmConfig:
    """A kvm_config for a workload shape.  With a host-resident repository the
    GPU reads missed blocks from pinned host memory itself (h2d_mode 1) unless
    h2d_mode=0 asks for copy-engine transfers.  candidate_mode=1 leaves sink and
    recent blocks out of the Eq. (10) softmax.  host_tier_blocks > 0 runs the
    host-tier policy (kvm_tier_step) over every step's selection.  index_spill=1
    makes a host-resident index cross the host link once per scoring call
    instead of once per pass; spill_tiles=m > 0 caps the tiles it keeps in
    device memory at m, and pass 2 re-streams the others."""
    mb = max_blocks if max_blocks is not None else wl.n_blocks + wl.steps * wl.append_blocks
    mp = max_positions if max_positions is not None else max(mb, wl.view_blocks) * BLOCK_TOKENS
    il = index_location if index_location is not None else (
        KVM_HOST_PINNED if wl.index_loc == "host" else KVM_DEVICE)
    rl = repo_location if repo_location is not None else (
        KVM_HOST_PINNED if wl.repo == "host" else KVM_DEVICE)
    return KvmConfig(
        n_layers=wl.n_layers, n_kv_heads=wl.n_kv_heads, n_q_heads=wl.n_q_heads,
        head_dim=wl.head_dim, block_tokens=BLOCK_TOKENS, rope_theta=wl.rope_theta,
        kv_dtype=_DT[wl.kv_dtype], index_dtype=_DT[wl.index_dtype], q_dtype=_DT[wl.q_dtype],
        sink_blocks=wl.sink_blocks, recent_blocks=wl.recent_blocks,
        view_blocks=wl.view_blocks, max_queries=max_queries or wl.n_queries, max_blocks=mb,
        max_positions=mp, tile_blocks=wl.tile_blocks,
        pool_pages=pool_pages if pool_pages is not None else wl.view_blocks + wl.append_blocks,
        index_location=il, repo_location=rl, h2d_batch_blocks=h2d_batch_blocks,
        h2d_mode=h2d_mode, score_variant=score_variant, delta_rerope_limit=delta_rerope_limit,
        candidate_mode=candidate_mode, host_tier_blocks=host_tier_blocks,
        host_tier_lambda=host_tier_lambda, index_spill=index_spill, spill_tiles=spill_tiles)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def score_select_static(cfg: KvmConfig, q, n_queries: int, index, n_blocks: int, scores_out,
                        sel_ids_out, stream=None) -> int:
    """kvm_score_select_static: scoring + selection for callers that cannot
    allocate device memory.  Needs no Context and no workspace; the library's
    fixed 32 MiB device scratch is used instead (calls must not overlap on the
    GPU).  Returns the number of selected blocks."""
    lib = load()
    n_sel = ctypes.c_int32()
    check(lib.kvm_score_select_static(ctypes.byref(cfg), _ptr(q), n_queries, _ptr(index),
                                      n_blocks, _ptr(scores_out), _ptr(sel_ids_out),
                                      ctypes.byref(n_sel), _stream(stream)),
          "kvm_score_select_static")
    return n_sel.value


def score_select_static_status(stream=None) -> None:
    """kvm_score_select_static_status: waits for ``stream`` and raises
    KvmError (KVM_ERR_TIMEOUT or KVM_ERR_DEVICE) when a device flag was raised
    by kvm_score_select_static calls since the last check; the flag is cleared."""
    check(load().kvm_score_select_static_status(_stream(stream)),
          "kvm_score_select_static_status")


def launch_count() -> int:
    """kvm_launch_count: kernels the library has launched in this process so
    far (the difference across a region counts the kernels it launched)."""
    return int(load().kvm_launch_count())


class HostTier:
    """kvm_tier: host-tier admission and eviction (LRFU over retrievals) of the
    block repository.  Host-only; needs no GPU."""

    def __init__(self, capacity_blocks: int, lam: float):
        self.lib = load()
        h = ctypes.c_void_p()
        check(self.lib.kvm_tier_create(int(capacity_blocks), float(lam), ctypes.byref(h)),
              "kvm_tier_create")
        self.handle = h

    def step(self, ids, n_blocks: int):
        """One step: returns (hits, misses, demoted ids in demotion order)."""
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        dem = np.empty(max(int(n_blocks), 1), dtype=np.int32)
        st = KvmTierStats()
        check(self.lib.kvm_tier_step(self.handle, arr.ctypes.data if arr.size else None,
                                     int(arr.size), int(n_blocks), dem.ctypes.data,
                                     ctypes.byref(st)), "kvm_tier_step")
        return st.hits, st.misses, dem[:st.demoted].tolist()

    def resident(self, n: int):
        import numpy as np
        flags = np.zeros(max(int(n), 1), dtype=np.uint8)
        check(self.lib.kvm_tier_resident(self.handle, flags.ctypes.data, int(n)),
              "kvm_tier_resident")
        return flags[:n]

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.kvm_tier_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepStats(Mapping):
    """The counters of one kvm_step, read from the kvm_step_stats the library
    fills (by the next kvm_sync at the latest)."""

    _KEYS = tuple(f for f, _ in KvmStepStats._fields_)

    def __init__(self, st: KvmStepStats):
        self._st = st

    def __getitem__(self, k):
        if k not in self._KEYS:
            raise KeyError(k)
        return getattr(self._st, k)

    def __iter__(self):
        return iter(self._KEYS)

    def __len__(self):
        return len(self._KEYS)


class Context:
    """A kvm_ctx plus its caller-owned device workspace (a torch uint8 tensor)."""

    def __init__(self, cfg: KvmConfig, device="cuda", stream=None):
        self.lib = load()
        self.cfg = cfg
        nbytes = self.lib.kvm_workspace_bytes(ctypes.byref(cfg))
        if nbytes == 0:
            raise KvmError(-1, "kvm_workspace_bytes", "invalid config")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        check(self.lib.kvm_create(ctypes.byref(cfg), self.workspace.data_ptr(), nbytes,
                                  _stream(stream), ctypes.byref(h)), "kvm_create")
        self.handle = h
        self._bound = None
        self._pending = []

    # -- shapes -----------------------------------------------------------
    @property
    def kv_dtype(self) -> torch.dtype:
        return _TDT[self.cfg.kv_dtype]

    @property
    def index_dtype(self) -> torch.dtype:
        return _TDT[self.cfg.index_dtype]

    def block_shape(self, n: int):
        c = self.cfg
        return (n, c.n_layers, c.n_kv_heads, BLOCK_TOKENS, c.head_dim)

    def index_shape(self):
        c = self.cfg
        return (c.n_layers, c.n_kv_heads, c.max_blocks, c.head_dim)

    # -- the four calls -----------------------------------------------------
    def build_index(self, k_pages, first_block: int, n_blocks: int, index, raw_k_out=None,
                    stream=None) -> None:
        check(self.lib.kvm_build_index(self.handle, _ptr(k_pages), first_block, n_blocks,
                                       _ptr(index), _ptr(raw_k_out), _stream(stream)),
              "kvm_build_index")

    def score_select(self, q, n_queries: int, index, n_blocks: int, scores_out, sel_ids_out,
                     stream=None) -> int:
        n_sel = ctypes.c_int32()
        check(self.lib.kvm_score_select(self.handle, _ptr(q), n_queries, _ptr(index), n_blocks,
                                        _ptr(scores_out), _ptr(sel_ids_out),
                                        ctypes.byref(n_sel), _stream(stream)),
              "kvm_score_select")
        return n_sel.value

    def assemble_view(self, sel_ids, page_ids, n_sel: int, raw_k_repo, v_repo, k_pages,
                      v_pages, stream=None) -> None:
        check(self.lib.kvm_assemble_view(self.handle, _ptr(sel_ids), _ptr(page_ids), n_sel,
                                         _ptr(raw_k_repo), _ptr(v_repo), _ptr(k_pages),
                                         _ptr(v_pages), _stream(stream)),
              "kvm_assemble_view")

    def bind(self, *, index, raw_k, v, pool_k, pool_v, page_table, scores, sel_ids,
             pool_raw_k=None) -> None:
        b = KvmBuffers(index=_ptr(index), raw_k=_ptr(raw_k), v=_ptr(v), pool_k=_ptr(pool_k),
                       pool_v=_ptr(pool_v), pool_raw_k=_ptr(pool_raw_k),
                       page_table=_ptr(page_table), scores=_ptr(scores), sel_ids=_ptr(sel_ids))
        check(self.lib.kvm_bind(self.handle, ctypes.byref(b)), "kvm_bind")
        self._bound = dict(index=index, raw_k=raw_k, v=v, pool_k=pool_k, pool_v=pool_v,
                           pool_raw_k=pool_raw_k, page_table=page_table, scores=scores,
                           sel_ids=sel_ids)

    def stage_out(self, raw_k, v, first_block: int, n_blocks: int, stream=None) -> None:
        """kvm_stage_out: copy completed blocks' raw K / V into the bound host
        repository, overlapped with later work on `stream`."""
        check(self.lib.kvm_stage_out(self.handle, _ptr(raw_k), _ptr(v), first_block, n_blocks,
                                     _stream(stream)), "kvm_stage_out")

    def reset_pool(self) -> None:
        check(self.lib.kvm_reset_pool(self.handle), "kvm_reset_pool")

    def step(self, q, n_queries: int, n_blocks: int, stream=None, stats=None):
        """One kvm_step.  The returned counters are final once sync() returns
        (a step whose residency diff runs on the device fills them then).
        With stats=False, or by default while the current stream is being
        captured into a CUDA graph, no counters are kept and None is returned."""
        if stats is None:
            stats = not (torch.cuda.is_available() and torch.cuda.is_current_stream_capturing())
        if not stats:
            check(self.lib.kvm_step(self.handle, _ptr(q), n_queries, n_blocks, None,
                                    _stream(stream)), "kvm_step")
            return None
        st = KvmStepStats()
        check(self.lib.kvm_step(self.handle, _ptr(q), n_queries, n_blocks, ctypes.byref(st),
                                _stream(stream)), "kvm_step")
        self._pending.append(st)           # the library writes it until the next sync
        return StepStats(st)

    def graph_step_stats(self, stream=None) -> "StepStats":
        """The counters of the last kvm_step launched from a CUDA graph on this
        context (waits for `stream`)."""
        st = KvmStepStats()
        check(self.lib.kvm_graph_step_stats(self.handle, ctypes.byref(st), _stream(stream)),
              "kvm_graph_step_stats")
        return StepStats(st)

    def sync(self, stream=None) -> None:
        check(self.lib.kvm_sync(self.handle, _stream(stream)), "kvm_sync")
        self._pending.clear()

    def debug_inject(self, what: int, nth: int) -> None:
        check(self.lib.kvm_debug_inject(self.handle, what, nth), "kvm_debug_inject")

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.lib.kvm_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
