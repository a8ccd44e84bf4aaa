"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi's CSV (a stand-in nvidia-smi on PATH prints fixed rows), the
step-byte count of the default workload, and the reference arm's JSON line."""
import os
import stat
import sys
import time

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _fake_smi(tmp_path, rows):
    d = tmp_path / "bin"
    d.mkdir()
    f = d / "nvidia-smi"
    body = "".join(f'echo "{r}"; ' for r in rows)
    f.write_text(f"#!/bin/bash\nwhile true; do {body}sleep 0.02; done\n")
    f.chmod(f.stat().st_mode | stat.S_IEXEC)
    return str(d)


@pytest.mark.parametrize("rows,median,reasons", [
    (["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"], 2070.0, []),
    (["0, 1500, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
      "0, 1700, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"], 1600.0, ["sw_power_cap"]),
    (["0, 900, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active"], 900.0, ["hw_slowdown"]),
])
def test_clock_sampler_parses_nvidia_smi_rows(tmp_path, monkeypatch, rows, median, reasons):
    import bench
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks(0)
    c.start()
    time.sleep(0.3)
    out = c.stop()
    assert out["samples"] >= 2
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == pytest.approx(median)
    assert out["reasons"] == reasons


def test_clock_sampler_without_nvidia_smi(monkeypatch, tmp_path):
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.Clocks(0)
    c.start()
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_step_bytes_weights_match_the_published_parameter_count():
    """The weight part of the roofline's algorithmic bytes (BF16, one request) is the
    drafter checkpoint's published parameter count (LSE docs/DFLASH2.md, compatible
    drafter paragraph) in BF16, without the two codebooks (only the gathered rows are
    read) and without the norm and conv-base vectors (not counted), plus the shared
    BF16 LM head, which the checkpoint does not hold."""
    import json
    import bench
    import workloads as wk
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "lse_dflash2_facts.json")))
    wl = wk.workload(2)
    g = wl.geom
    H, V, r = g.hidden, g.vocab, g.rank
    assert (H, g.n_layers, V, r) == (5120, 5, 248320, 256)
    kv = (min(wl.ctx[0], g.window - 1) + 8) * 2 * g.kv_dim * 2 * g.n_layers
    extra = kv + 8 * g.n_taps * H * 4 + 8 * V * 4 + (1 + 6 * 16 + 7 * 16) * r * 2
    weights = bench.step_bytes(wl, 1) - extra
    expected = 2 * (gold["bf16_params"] - 2 * V * r) + 2 * V * H
    # what is left out: the checkpoint's vectors (norm weights, conv bases), whose
    # shapes the input generators' table gives (a table the oracle pins test ties to the same count)
    from workloads.gen import weight_shapes
    shp = weight_shapes(wk.FULL)
    vec_params = sum(int(np.prod(s)) for k, s in shp.items()
                     if k not in ("embed", "lm_head") and not (len(s) == 2 and k.split(".")[-1] in wk.MATRIX_NAMES))
    assert expected - weights == 2 * vec_params


def test_reference_arm_prints_the_contract_line(capsys):
    """`bench.py --impl reference` on rank 0: one JSON line with the arm's keys, the
    oracle timed on the host (toy workload, one step)."""
    import json
    import bench
    args = bench.parse(["--impl", "reference", "--config", "1", "--steps", "1", "--warmup", "0"])
    bench.main_reference(args, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "steps/s"
    assert line["value"] > 0 and line["steps"] == 1 and line["n_gpus"] == 1 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "cfg1_toy"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
