"""ctypes declarations of the C ABI in include/kvm.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkvm.so")

KVM_F32, KVM_BF16, KVM_E4M3 = 0, 1, 2
KVM_DEVICE, KVM_HOST_PINNED = 0, 1

STATUS = {
    0: "KVM_OK", -1: "KVM_ERR_INVALID_ARG", -2: "KVM_ERR_WORKSPACE_TOO_SMALL",
    -3: "KVM_ERR_CAPACITY", -4: "KVM_ERR_CUDA", -5: "KVM_ERR_TIMEOUT",
    -6: "KVM_ERR_NOT_BOUND", -7: "KVM_ERR_INJECTED", -8: "KVM_ERR_DEVICE",
}


class KvmConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("n_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_tokens", ctypes.c_int32), ("rope_theta", ctypes.c_double),
        ("kv_dtype", ctypes.c_int32), ("index_dtype", ctypes.c_int32),
        ("q_dtype", ctypes.c_int32), ("sink_blocks", ctypes.c_int32),
        ("recent_blocks", ctypes.c_int32), ("view_blocks", ctypes.c_int32),
        ("max_queries", ctypes.c_int32), ("max_blocks", ctypes.c_int64),
        ("max_positions", ctypes.c_int64), ("tile_blocks", ctypes.c_int32),
        ("pool_pages", ctypes.c_int32), ("index_location", ctypes.c_int32),
        ("repo_location", ctypes.c_int32), ("h2d_batch_blocks", ctypes.c_int32),
        ("h2d_mode", ctypes.c_int32), ("score_variant", ctypes.c_int32),
        ("delta_rerope_limit", ctypes.c_int32), ("candidate_mode", ctypes.c_int32),
        ("host_tier_blocks", ctypes.c_int64), ("host_tier_lambda", ctypes.c_double),
        ("index_spill", ctypes.c_int32), ("spill_tiles", ctypes.c_int32),
    ]


class KvmBuffers(ctypes.Structure):
    _fields_ = [
        ("index", ctypes.c_void_p), ("raw_k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("pool_k", ctypes.c_void_p), ("pool_v", ctypes.c_void_p),
        ("pool_raw_k", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("scores", ctypes.c_void_p), ("sel_ids", ctypes.c_void_p),
    ]


class KvmStepStats(ctypes.Structure):
    _fields_ = [
        ("n_blocks", ctypes.c_int64), ("n_sel", ctypes.c_int32), ("hits", ctypes.c_int32),
        ("misses", ctypes.c_int32), ("reroped", ctypes.c_int32), ("evicted", ctypes.c_int32),
        ("h2d_copies", ctypes.c_int32), ("h2d_bytes", ctypes.c_int64),
        ("delta_reroped", ctypes.c_int32), ("host_hits", ctypes.c_int32),
        ("host_misses", ctypes.c_int32), ("host_demoted", ctypes.c_int32),
    ]


class KvmTierStats(ctypes.Structure):
    _fields_ = [
        ("hits", ctypes.c_int32), ("misses", ctypes.c_int32), ("demoted", ctypes.c_int32),
        ("resident", ctypes.c_int64),
    ]


# name -> (restype, argtypes)
SIGNATURES = {
    "kvm_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(KvmConfig)]),
    "kvm_create": (ctypes.c_int, [ctypes.POINTER(KvmConfig), ctypes.c_void_p, ctypes.c_size_t,
                                  ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "kvm_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "kvm_build_index": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p]),
    "kvm_score_select": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
                                        ctypes.c_void_p]),
    "kvm_assemble_view": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvm_bind": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(KvmBuffers)]),
    "kvm_reset_pool": (ctypes.c_int, [ctypes.c_void_p]),
    "kvm_stage_out": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "kvm_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                ctypes.c_int64, ctypes.POINTER(KvmStepStats), ctypes.c_void_p]),
    "kvm_score_select_static": (ctypes.c_int, [ctypes.POINTER(KvmConfig), ctypes.c_void_p,
                                               ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                               ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.POINTER(ctypes.c_int32), ctypes.c_void_p]),
    "kvm_score_select_static_status": (ctypes.c_int, [ctypes.c_void_p]),
    "kvm_tier_create": (ctypes.c_int, [ctypes.c_int64, ctypes.c_double,
                                       ctypes.POINTER(ctypes.c_void_p)]),
    "kvm_tier_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                     ctypes.c_int64, ctypes.c_void_p,
                                     ctypes.POINTER(KvmTierStats)]),
    "kvm_tier_resident": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]),
    "kvm_tier_destroy": (ctypes.c_int, [ctypes.c_void_p]),
    "kvm_sync": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "kvm_graph_step_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "kvm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kvm_last_error": (ctypes.c_char_p, []),
    "kvm_debug_inject": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64]),
    "kvm_launch_count": (ctypes.c_int64, []),
    "kvm_host_alloc": (ctypes.c_int, [ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p)]),
    "kvm_host_free": (ctypes.c_int, [ctypes.c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvm.so and declare every entry point.  Raises if the library is
    missing: there is no fallback implementation."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libkvm.so not found at {path}; build it with "
            "`python -m paged_kv_cache_meank_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class KvmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {detail}")


def check(status: int, where: str) -> None:
    if status != 0:
        detail = load().kvm_last_error().decode(errors="replace")
        raise KvmError(status, where, detail)
