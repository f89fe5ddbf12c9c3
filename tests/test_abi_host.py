"""The C ABI library on the host: it loads, exports every entry point the
header declares, and rejects bad configurations before touching the GPU."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_meank_gb300 import _abi, config_for, configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvm.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvm_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        from paged_kv_cache_meank_gb300 import build
        build.build()
    return _abi.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "kvm_build_index" in names and "kvm_step" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi.SIGNATURES), (set(names) ^ set(_abi.SIGNATURES))


def test_status_strings(lib):
    for code in _abi.STATUS:
        assert lib.kvm_status_string(code)
    assert lib.kvm_status_string(0) == b"ok"


def test_workspace_bytes_and_validation(lib):
    cfg = config_for(configs.TINY)
    n = lib.kvm_workspace_bytes(ctypes.byref(cfg))
    assert n > cfg.max_positions * 32 * 8  # at least the cos/sin table
    for field, bad in [("head_dim", 96), ("block_tokens", 16), ("n_q_heads", 5),
                       ("view_blocks", 5), ("kv_dtype", 7), ("max_blocks", 0),
                       ("pool_pages", 1), ("max_queries", 1000), ("candidate_mode", 2),
                       ("delta_rerope_limit", -1), ("h2d_mode", 3), ("index_spill", 2),
                       ("spill_tiles", -1), ("spill_tiles", 3)]:   # 3 needs index_spill
        c = config_for(configs.TINY)
        setattr(c, field, bad)
        assert lib.kvm_workspace_bytes(ctypes.byref(c)) == 0, field
        h = ctypes.c_void_p()
        st = lib.kvm_create(ctypes.byref(c), None, 0, None, ctypes.byref(h))
        assert st == -1 and not h.value, field


def test_create_rejects_small_or_misaligned_workspace(lib):
    cfg = config_for(configs.TINY)
    n = lib.kvm_workspace_bytes(ctypes.byref(cfg))
    h = ctypes.c_void_p()
    # host-side checks fire before any CUDA call; the pointers are never dereferenced
    assert lib.kvm_create(ctypes.byref(cfg), ctypes.c_void_p(4096), n - 1, None,
                          ctypes.byref(h)) == -2
    assert lib.kvm_create(ctypes.byref(cfg), ctypes.c_void_p(4097), n, None,
                          ctypes.byref(h)) == -1
    assert b"aligned" in lib.kvm_last_error()


def test_calls_reject_null_context(lib):
    n0 = lib.kvm_launch_count()
    assert lib.kvm_build_index(None, None, 0, 0, None, None, None) == -1
    assert lib.kvm_score_select(None, None, 1, None, 1, None, None, None, None) == -1
    assert lib.kvm_assemble_view(None, None, None, 0, None, None, None, None, None) == -1
    assert lib.kvm_step(None, None, 1, 1, None, None) == -1
    assert lib.kvm_destroy(None) == 0
    assert lib.kvm_launch_count() == n0     # rejected on the host: no kernel launched


def test_layout_sizes_follow_the_workloads():
    # index footprint: 16 layers x 8 KV heads x 128 d x 2 B = 32 KiB per block, the
    # per-block index size the KVMem scaling table implies (0.25 GiB at 256K tokens)
    assert configs.W1M.index_entry_bytes == 32 * 1024
    assert configs.W256K.n_blocks * configs.W1M.index_entry_bytes == 256 * 1024 ** 2
    # KV bytes per block 2 * L * c * h * d * b (InferScale §4 storage cost) for c = 32
    w = configs.W256K
    assert 2 * w.block_bytes == 2 * w.n_layers * 32 * w.n_kv_heads * w.head_dim * 2


def test_index_spill_workspace_holds_the_index(lib):
    """With a host-resident index, index_spill keeps one staging tile per index
    tile in the workspace: it grows by the index size less the two tiles that
    the default double buffering needs."""
    wl = configs.W1M
    base = config_for(wl)
    spill = config_for(wl, index_spill=1)
    n0 = lib.kvm_workspace_bytes(ctypes.byref(base))
    n1 = lib.kvm_workspace_bytes(ctypes.byref(spill))
    tile = wl.n_layers * wl.n_kv_heads * base.tile_blocks * wl.head_dim * 2
    tiles = -(-base.max_blocks // base.tile_blocks)
    assert n1 - n0 == tiles * tile - 2 * tile
    # a budget of m tiles: two streaming tiles and m kept ones; a budget of
    # the whole index or more is the full spill
    for m in (1, 5):
        capped = config_for(wl, index_spill=1, spill_tiles=m)
        assert lib.kvm_workspace_bytes(ctypes.byref(capped)) - n0 == m * tile
    for m in (tiles, tiles + 7):
        whole = config_for(wl, index_spill=1, spill_tiles=m)
        assert lib.kvm_workspace_bytes(ctypes.byref(whole)) == n1
    # a device-resident index stages nothing either way
    dev = config_for(wl, index_location=0)
    dev_spill = config_for(wl, index_location=0, index_spill=1)
    assert lib.kvm_workspace_bytes(ctypes.byref(dev)) == lib.kvm_workspace_bytes(
        ctypes.byref(dev_spill))


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of kvm_config, kvm_buffers, kvm_step_stats and
    kvm_tier_stats have the header's sizes and field offsets (a C program
    compiled against include/kvm.h prints them)."""
    import os
    import shutil
    import subprocess
    from paged_kv_cache_meank_gb300 import _abi
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"kvm_config": _abi.KvmConfig, "kvm_buffers": _abi.KvmBuffers,
               "kvm_step_stats": _abi.KvmStepStats, "kvm_tier_stats": _abi.KvmTierStats}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kvm.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run([cc, "-std=c99", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)
