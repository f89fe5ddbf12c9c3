"""The bench's roofline arithmetic, on the host: the units of work per
(layer, kv head, block) that each line divides by, which unit binds, and the
DRAM traffic taken from the committed ncu summaries only while the kernel
sources match them."""
import json
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from paged_kv_cache_meank_gb300 import configs  # noqa: E402


@pytest.fixture
def gb300(monkeypatch):
    """The one CUDA query the roofline makes (the SM count), answered as on GB300."""
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda dev: types.SimpleNamespace(multi_processor_count=152))


class _Step:
    pass


def test_scoring_line_is_bound_by_the_tensor_pipe(gb300):
    """10M-token scoring alone: per (layer, kv head, block) two exact passes
    take 2 x 2*d*rows flops, 2*rows exponentials and one 256-byte index read;
    the tensor floor is the highest, so it is the roofline, with HBM (one
    read) and MUFU (32 ex2 per clock per SM) beside it."""
    wl = configs.ALL["q27-10m-score"]
    ms = 14.2
    comps, roof = bench.summarize(wl, _Step(), ms, {"score_select": ms},
                                  {"sm_max_mhz": 2070.0}, None, None)
    units = 312500 * 64 * 8
    rows = 32 * 6
    flops = 2 * (2 * 128 * rows) * units
    assert flops == 98304 * units
    burst, sustained, _ = bench._bf16_peaks()
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["algorithmic_flops"] == flops
    assert roof["achieved"] == pytest.approx(flops / (ms * 1e-3) / 1e12)
    assert roof["peak"] == sustained and roof["frac"] == pytest.approx(roof["achieved"] / sustained)
    assert roof["frac_burst"] == pytest.approx(roof["achieved"] / burst)
    hbm = roof["hbm"]
    assert hbm["algorithmic_bytes"] == units * 256            # the index, read once
    assert hbm["frac"] == pytest.approx(units * 256 / (ms * 1e-3) / 1e9 / bench._peaks()[0])
    mufu = roof["mufu"]
    assert mufu["algorithmic_ops"] == 2 * rows * units
    assert mufu["peak"] == pytest.approx(32 * 152 * 2070.0 * 1e-3)
    # at these sizes the tensor floor is above the MUFU and one-read HBM floors
    t_tensor = flops / (sustained * 1e12)
    t_mufu = mufu["algorithmic_ops"] / (mufu["peak"] * 1e9)
    t_hbm = hbm["algorithmic_bytes"] / (bench._peaks()[0] * 1e9)
    assert t_tensor > max(t_mufu, t_hbm)
    assert comps["score_blocks_per_s"] == pytest.approx(312500 / (ms * 1e-3))


def test_default_step_line_is_the_build_against_hbm(gb300):
    """The 256K step: the build dominates, at 32*d*2 bytes of K in, as many
    of raw K out and d*2 of Mean-K out per (layer, kv head, block)."""
    wl = configs.W256K
    parts = {"build": 10.37, "score_select": 0.45, "assemble": 2.53}
    comps, roof = bench.summarize(wl, _Step(), sum(parts.values()), parts,
                                  {"sm_max_mhz": 2070.0}, None, None)
    units = 8192 * 64 * 8
    assert roof["bound"] == "hbm" and roof["kernel"] == "build"
    assert roof["algorithmic_bytes"] == units * 16640
    assert roof["frac"] == pytest.approx(units * 16640 / (10.37e-3) / 1e9 / bench._peaks()[0])
    view_tokens = 1024 * 32
    assert comps["kernels"]["assemble"]["gbs"] == pytest.approx(
        view_tokens * 4 * 64 * 8 * 128 * 2 / 2.53e-3 / 1e9)
    # the whole step with the index read twice, over the step time
    step_bytes = units * 16640 + 2 * units * 256 + view_tokens * 4 * 64 * 8 * 128 * 2
    assert comps["step_hbm_frac"] == pytest.approx(
        step_bytes / (sum(parts.values()) * 1e-3) / 1e9 / bench._peaks()[0])


def test_traffic_is_used_only_while_the_sources_match(tmp_path, monkeypatch):
    """A traffic entry counts while every listed source hashes as recorded;
    a changed source voids it."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        entry = json.load(f)["q27-256k"]["build"]
    assert bench._traffic_from_profile("q27-256k", "build") == entry["bytes"]
    # the same entry over a copy of the source with one byte changed
    root = tmp_path / "repo"
    (root / "profiles").mkdir(parents=True)
    src = root / entry["source"]
    src.parent.mkdir(parents=True)
    with open(os.path.join(ROOT, entry["source"]), "rb") as f:
        data = f.read()
    src.write_bytes(data)
    (root / "profiles" / "traffic.json").write_text(json.dumps({"w": {"build": entry}}))
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench._traffic_from_profile("w", "build") == entry["bytes"]
    src.write_bytes(data + b" ")
    assert bench._traffic_from_profile("w", "build") is None
    assert bench._traffic_from_profile("w", "assemble") is None
