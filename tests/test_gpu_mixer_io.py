"""kda_premix and kda_output_gate on the GPU against the fp64 oracle, element by element.

Bounds, from the arithmetic (fp32 in the kernels, fp64 in the oracle, the same inputs):
  - bf16 outputs are the fp32 result rounded to nearest: |gpu - ref| <= 2^-8 |ref| plus the fp32
    error of the 4-tap sums, which can cancel (atol 1e-5 on O(1) data);
  - fp32 outputs: a few fp32 ulps of the terms (rtol 2e-6, atol 2e-6).
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
BOUND = {"bf16": (2.0 ** -8, 1e-5), "f32": (2e-6, 2e-6)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    yield
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def assert_elementwise(name, gpu, ref, dtype):
    rtol, atol = BOUND[dtype]
    g = gpu.detach().to("cpu", torch.float64).numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    excess = np.abs(g - ref) - (rtol * np.abs(ref) + atol)
    worst = int(np.argmax(excess)) if excess.size else 0
    assert excess.size == 0 or excess.flat[worst] <= 0, (
        f"{name}: element {np.unravel_index(worst, g.shape)} gpu {g.flat[worst]!r} "
        f"oracle {ref.flat[worst]!r}")


def run_premix(orc, x, dtype, heads=None):
    """GPU pre-mixer on x (device tensors) and the oracle on the same inputs (optionally on a
    subset of heads); returns the GPU outputs."""
    out = kda.premix(x["xq"], x["xk"], x["xv"], x["a"], x["b"], x["w"], x["cu_seqlens"], x["hist"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    H, d = x["xq"].shape[1:]
    hs = list(range(H)) if heads is None else list(heads)
    idx = torch.tensor(hs, device=DEV)
    cols = (idx[:, None] * d + torch.arange(d, device=DEV)).reshape(-1)
    sel = lambda t: t.index_select(1, idx).cpu()
    hist = None if x["hist"] is None else x["hist"].index_select(3, cols).cpu()
    ref = orc.premix(sel(x["xq"]), sel(x["xk"]), sel(x["xv"]), sel(x["a"]), sel(x["b"]),
                     x["w"].index_select(1, cols).cpu(), hist=hist,
                     cu_seqlens=x["cu_seqlens"].cpu().long())
    for name, got, want in zip(("q", "k", "v", "g", "beta"), out, ref):
        assert_elementwise(name, got.index_select(1, idx), want, dtype)
    return out


@pytest.mark.parametrize("dtype,lengths,H,d,hist", [
    ("bf16", [100, 1, 37, 2, 64], 3, 128, False),
    ("bf16", [100, 1, 37, 2, 64], 3, 128, True),
    ("bf16", [31, 32, 33], 4, 128, True),
    ("bf16", [127, 1, 129, 3], 2, 128, True),       # sequence edges next to 128-token boundaries
    ("bf16", [255, 1, 257, 3], 2, 128, True),       # sequence edges next to 256-token chunk edges
    ("bf16", [253, 6, 300], 3, 128, True),          # a sequence starting exactly at a chunk's halo
    ("bf16", [254, 5, 300], 3, 128, True),          # a sequence start inside a chunk's 3-token halo
    ("bf16", [0, 5, 0, 40, 0], 2, 128, True),       # empty sequences
    ("f32", [45, 3, 70], 5, 64, True),              # 320 channels: a partial channel block
    ("f32", [9], 2, 8, False),
    ("f32", [33], 1, 16, True),
    ("f32", [40, 40], 3, 32, True),
    ("f32", [17, 2], 9, 256, True),                 # 2304 channels: three channel blocks
    # bf16 with H*d a multiple of 1024 (whole channel blocks)
    ("bf16", [100, 1, 37, 2, 64], 8, 128, False),
    ("bf16", [255, 1, 257, 3], 8, 128, True),       # sequence edges next to chunk edges
    ("bf16", [0, 5, 0, 40, 0], 16, 64, True),       # empty sequences
    ("bf16", [300], 4, 256, True),                  # last chunk of 44 tokens: a partial prefetch group
    ("bf16", [77, 200], 32, 64, False),             # two channel blocks
    ("bf16", [20, 13], 128, 8, True),               # one thread per head
])
def test_premix_parity(orc, dtype, lengths, H, d, hist):
    x = synth.make_premix_inputs(lengths, heads=H, d=d, dtype=dtype, seed=sum(lengths) + H + d,
                                 device=DEV, hist=hist)
    run_premix(orc, x, dtype)


def test_premix_full_size_sampled_heads(orc):
    # T = 8192, H = 96, d = 128 in one launch; the oracle checks 8 heads spread over the range
    x = synth.make_premix_inputs([8192], dtype="bf16", seed=61, device=DEV)
    run_premix(orc, x, "bf16", heads=[0, 13, 31, 47, 64, 80, 94, 95])


def test_premix_varlen8_with_history(orc):
    x = synth.make_premix_inputs(synth.varlen8_lengths(), dtype="bf16", seed=62, device=DEV, hist=True)
    run_premix(orc, x, "bf16", heads=[5, 77])


def test_premix_no_tokens():
    x = synth.make_premix_inputs([0], heads=2, d=128, dtype="bf16", device=DEV)
    out = kda.premix(x["xq"], x["xk"], x["xv"], x["a"], x["b"], x["w"])
    torch.cuda.synchronize()
    assert all(t.numel() == 0 for t in out)


def test_premix_feeds_prefill(orc):
    # the pre-mixer's outputs drive the recurrence: GPU premix -> prefill against the oracle's
    # premix -> prefill on the same projections (bf16 inputs, fp32 state)
    lengths = [200, 57]
    x = synth.make_premix_inputs(lengths, heads=2, d=128, dtype="bf16", seed=63, device=DEV, hist=True)
    q, k, v, g, beta = kda.premix(x["xq"], x["xk"], x["xv"], x["a"], x["b"], x["w"],
                                  x["cu_seqlens"], x["hist"])
    out, fin, _ = kda.prefill(q, k, v, g, beta, x["cu_seqlens"], lengths=lengths)
    torch.cuda.synchronize()
    cpu = {k_: (t.cpu() if t is not None and hasattr(t, "cpu") else t) for k_, t in x.items()}
    ref = orc.premix(cpu["xq"], cpu["xk"], cpu["xv"], cpu["a"], cpu["b"], cpu["w"],
                     hist=cpu["hist"], cu_seqlens=cpu["cu_seqlens"].long())
    # the recurrence's inputs travel as bf16 on both sides (the pre-mixer's output dtype)
    rq, rk, rv, rg, rb = (torch.from_numpy(r).to(torch.bfloat16) for r in ref)
    ro, rf, _ = orc.prefill(rq, rk, rv, rg, rb, cpu["cu_seqlens"].long())
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final_state", fin, rf, TOL["bf16"]["state"])


@pytest.mark.parametrize("o_dt,z_dt,out_dt", [
    (o, z, y) for o in ("f32", "bf16") for z in ("f32", "bf16") for y in ("f32", "bf16")])
def test_output_gate_parity(orc, o_dt, z_dt, out_dt):
    for shape in ((37, 3, 128), (13, 7)):           # the second is not a multiple of 8 elements
        x = synth.make_gate_inputs(shape, o_dt, z_dt, seed=len(shape), device=DEV)
        out = kda.output_gate(x["o"], x["z"], out_dtype=synth.torch_dtype(out_dt))
        torch.cuda.synchronize()
        ref = orc.output_gate(x["o"].cpu(), x["z"].cpu())
        assert_elementwise("out", out, ref, out_dt)


def test_output_gate_in_place_and_empty(orc):
    x = synth.make_gate_inputs((64, 96, 128), "f32", "bf16", seed=5, device=DEV)
    ref = orc.output_gate(x["o"].cpu(), x["z"].cpu())
    o = x["o"]
    res = kda.output_gate(o, x["z"], out=o)
    torch.cuda.synchronize()
    assert res.data_ptr() == o.data_ptr()
    assert_elementwise("in place", o, ref, "f32")
    e = synth.make_gate_inputs((0, 128), "f32", "f32", device=DEV)
    assert kda.output_gate(e["o"], e["z"]).numel() == 0


def test_output_gate_full_size(orc):
    # the T = 8192, H = 96 output: fp32 o, bf16 gate pre-activation, bf16 result
    x = synth.make_gate_inputs((8192, 96, 128), "f32", "bf16", seed=6, device=DEV)
    out = kda.output_gate(x["o"], x["z"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 4095, 8190, 8191], device=DEV)
    ref = orc.output_gate(x["o"][rows].cpu(), x["z"][rows].cpu())
    assert_elementwise("out", out[rows], ref, "bf16")
