"""libkvm from a plain C program (tests/c_client/kvm_client.c): no Python, no
PyTorch, device memory from cudaMalloc, every step through the C ABI.  The CPU
test compiles and links the client against the header and the library; the GPU
test runs it on the tiny workload and checks its outputs against the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle.kvmem as ora
from gpu_helpers import assert_meank_close, assert_scores_close, assert_storage_close
from paged_kv_cache_meank_gb300 import _abi, configs, workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "kvm_client.c")
PKG = os.path.dirname(_abi.LIB_PATH)


def _compile(tmp_path) -> str:
    if not os.path.exists(_abi.LIB_PATH):
        from paged_kv_cache_meank_gb300 import build
        build.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "kvm_client")
    cmd = [nvcc, "-O2", "-I" + os.path.join(ROOT, "include"), SRC, "-o", exe,
           "-L" + PKG, "-lkvm", "-Xlinker", "-rpath=" + PKG]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_client_recall_step_matches_oracle(tmp_path):
    wl = configs.TINY
    N, V, L, G, H, d = (wl.n_blocks, wl.view_blocks, wl.n_layers, wl.n_kv_heads,
                        wl.n_q_heads, wl.head_dim)
    exe = _compile(tmp_path)
    ws = workload.make_workspace(wl, seed=0)
    raw = ws.raw_k.numpy().astype(np.float32)
    # K as a prefill writes it: raw K rotated at original positions (oracle, float32)
    kp = np.empty_like(raw)
    pos = ora.block_positions(np.arange(N))
    for i in range(N):
        c, s = ora.cos_sin_f32(pos[i], d, wl.rope_theta)
        kp[i] = ora.rope_f32(raw[i], c, s)
    v = ws.v.numpy().astype(np.float32)
    q = ws.q.numpy().astype(np.float32)
    kp.tofile(tmp_path / "kpages.bin")
    v.tofile(tmp_path / "v.bin")
    q.tofile(tmp_path / "q.bin")
    args = [exe, str(tmp_path), L, G, H, d, repr(wl.rope_theta), N, wl.n_queries,
            wl.sink_blocks, wl.recent_blocks, V]
    r = subprocess.run([str(a) for a in args], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr

    def out(name, dtype, shape):
        return np.fromfile(tmp_path / name, dtype=dtype).reshape(shape)

    blk = (L, G, 32, d)
    index = out("index.bin", np.float32, (L, G, N, d))
    mk = ora.meank(kp, "f32", 0, wl.rope_theta)
    rms = float(np.sqrt(np.mean(raw.astype(np.float64) ** 2)))
    assert_meank_close(index, mk, "f32", rms, "C client index")
    raw_ref = ora.raw_k(kp, "f32", 0, wl.rope_theta)
    assert_storage_close(out("raw.bin", np.float32, (N,) + blk), raw_ref, "f32", "C client raw K")
    R = ora.block_relevance(q.astype(np.float64), mk.astype(np.float32).astype(np.float64), N)
    assert_scores_close(out("scores.bin", np.float32, (N,)), R, "C client scores")
    want = ora.select_blocks(R, wl.sink_blocks, wl.recent_blocks, V)
    sel = out("sel.bin", np.int32, (V,))
    assert np.array_equal(sel, want), (sel, want)
    ref_k = ora.view_k(raw_ref[want], "f32", wl.rope_theta)
    assert_storage_close(out("pool_k.bin", np.float32, (V,) + blk), ref_k, "f32", "C client view K")
    assert np.array_equal(out("pool_v.bin", np.float32, (V,) + blk), v[want])
