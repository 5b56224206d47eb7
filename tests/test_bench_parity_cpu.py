"""The benchmark's CPU leg: it runs the oracle on the timed step's own inputs and compares the
step's results with it.  Checked on a shrunken workload with the oracle's own result standing in
for the GPU's: near-exact results pass, a planted error fails, and a sample shorter than the
sequence compares the outputs only."""
import numpy as np
import pytest
import torch

import bench
import oracle
from kimi_delta_attention_13_gb300 import synth


@pytest.fixture
def small(monkeypatch):
    monkeypatch.setattr(bench, "T1", 128)
    monkeypatch.setattr(bench, "H", 2)
    x = synth.make_inputs([128], heads=2, dtype="bf16", seed=1, device="cpu")
    o, f, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"])
    return {"inputs": {k: x[k] for k in ("q", "k", "v", "g", "beta")},
            "out": torch.from_numpy(o).float(), "final": torch.from_numpy(f).float()}


def test_parity_leg_passes_and_fails(small):
    base, parity = bench.cpu_baseline(small, target_s=5.0)
    assert base["kind"] == "oracle" and base["value"] > 0 and base["cores"] >= 1
    assert parity["tokens"] == 128 and parity["pass"]
    assert parity["out"] < 1e-6 and parity["final_state"] < 1e-6      # fp32 copies of the oracle
    small["out"][5, 1, 17] += 0.5                                       # one planted error
    _, parity = bench.cpu_baseline(small, target_s=5.0)
    assert not parity["pass"] and parity["out"] > bench.TOL_OUT


def test_short_sample_compares_outputs_only(small, monkeypatch):
    monkeypatch.setattr(bench, "T1", 256)     # the sample (128 tokens) no longer covers the sequence
    small["inputs"] = {k: torch.cat([t, t]) for k, t in small["inputs"].items()}
    small["out"] = torch.cat([small["out"], small["out"]])
    base, parity = bench.cpu_baseline(small, target_s=1e-6)   # bounded: 64 tokens
    assert parity["tokens"] == 64 and parity["final_state"] is None and parity["pass"]


def test_rel_err_metric():
    ref = np.array([3.0, -4.0])                                  # RMS = sqrt(12.5)
    assert bench.rel_err(ref + np.array([0.0, 0.5]), ref) == pytest.approx(0.5 / np.sqrt(12.5))
    assert bench.rel_err(np.zeros(0), np.zeros(0)) == 0.0


def test_other_workloads_parity_leg():
    # a kept head sample (varlen, initial states, checkpoints) with the oracle's own results as
    # the GPU's: it passes; a planted error in a checkpoint fails it; the kept data is dropped
    lengths, stride = [70, 0, 130], 32
    x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=3, device="cpu", init_state=True)
    cu = x["cu_seqlens"].long()
    o, f, c = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, x["state"],
                                       ckpt_stride=stride)
    check = {"heads": [0, 1], "ckpt_stride": stride,
             "inputs": {k: x[k] for k in ("q", "k", "v", "g", "beta")}, "cu": cu, "init": x["state"],
             "out": torch.from_numpy(o).float(), "final": torch.from_numpy(f).float(),
             "ckpts": torch.from_numpy(c).float()}
    named = {"w": {"ms": 1.0, "_check": check}}
    bench.other_parity(named)
    par = named["w"]["parity"]
    assert "_check" not in named["w"] and par["pass"] and par["ckpts"] < 1e-6
    check["ckpts"][1, 0, 3, 4] += 1.0
    named = {"w": {"ms": 1.0, "_check": check}}
    bench.other_parity(named)
    assert not named["w"]["parity"]["pass"] and named["w"]["parity"]["ckpts"] > bench.TOL_STATE
