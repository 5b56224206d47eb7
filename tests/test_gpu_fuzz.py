"""Seeded random cases of the prefill against the fp64 oracle: varlen batches whose lengths sit on
and around the 16-token tiles and 32-token steps (and random ones), 1 to 5 heads, with or without
initial states, checkpoint strides 0/32/64/96, fp32 or bf16 outputs, the default and the precise
build; seeded random decode batches; the staged prefill from pinned host buffers with random chunk
sizes; and the context-parallel prefill with random segment lengths.  Bounds as everywhere (bf16
inputs: 2e-2 x RMS on outputs, 1e-2 on states and checkpoints; bf16 outputs add their own
rounding, 2^-8 relative)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
EDGE = [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 95, 96, 97]


def cases(n=64, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        n_seqs = int(rng.integers(1, 6))
        lengths = [int(rng.choice(EDGE)) if rng.random() < 0.6 else int(rng.integers(1, 400))
                   for _ in range(n_seqs)]
        out.append(dict(lengths=lengths, heads=int(rng.integers(1, 6)),
                        init=bool(rng.random() < 0.5), stride=int(rng.choice([0, 32, 64, 96])),
                        bf16_out=bool(rng.random() < 0.3), precise=bool(rng.random() < 0.4),
                        seed=1000 + i))
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    yield
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("c", cases(), ids=lambda c: f"L{c['lengths']}-H{c['heads']}-s{c['stride']}"
                         f"{'-init' if c['init'] else ''}{'-bf16' if c['bf16_out'] else ''}"
                         f"{'-precise' if c['precise'] else ''}")
def test_fuzz_prefill(orc, c):
    x = synth.make_inputs(c["lengths"], heads=c["heads"], dtype="bf16", seed=c["seed"], device=DEV,
                          init_state=c["init"])
    odt = torch.bfloat16 if c["bf16_out"] else torch.float32
    out, fin, ck = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                               ckpt_stride=c["stride"], lengths=c["lengths"], out_dtype=odt,
                               precise=c["precise"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rf, rc = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu().long(),
                             x["state"], ckpt_stride=c["stride"])
    if c["bf16_out"]:
        g = out.double().cpu().numpy()
        rms = float(np.sqrt(np.mean(ro ** 2))) if ro.size else 0.0
        assert np.all(np.abs(g - ro) <= TOL["bf16"]["out"] * rms + 2.0 ** -8 * np.abs(ro))
    else:
        assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final", fin, rf, TOL["bf16"]["state"])
    if c["stride"]:
        n_ck = kda.num_checkpoints(c["lengths"], c["stride"])
        assert (ck.shape[0] if ck is not None else 0) == n_ck
        if n_ck:
            assert_close("ckpts", ck, rc, TOL["bf16"]["state"])


@pytest.mark.parametrize("i", range(8))
def test_fuzz_decode(orc, i):
    rng = np.random.default_rng(3000 + i)
    N, H = int(rng.integers(1, 40)), int(rng.integers(1, 6))
    d = synth.make_decode_inputs(N, heads=H, seed=3000 + i, device=DEV)
    state0 = d["state"].clone()
    out = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rs = orc.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state0)
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("state", d["state"], rs, TOL["bf16"]["state"])


@pytest.mark.parametrize("i", range(8))
def test_fuzz_staged(orc, i):
    rng = np.random.default_rng(4000 + i)
    lengths = [int(rng.choice(EDGE)) if rng.random() < 0.5 else int(rng.integers(1, 500))
               for _ in range(int(rng.integers(1, 6)))]
    H = int(rng.integers(1, 5))
    chunk = int(rng.choice([32, 64, 96, 128, 160, 256]))
    x = synth.make_inputs(lengths, heads=H, dtype="bf16", seed=4000 + i, device=DEV,
                          init_state=bool(rng.random() < 0.5))
    h = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    h_out, fin, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], x["cu_seqlens"].cpu(),
                                       x["state"], chunk_tokens=chunk, static_tables=bool(i % 2))
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rf, _ = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu().long(),
                            x["state"])
    assert_close("out", h_out, ro, TOL["bf16"]["out"])
    assert_close("final", fin, rf, TOL["bf16"]["state"])


@pytest.mark.parametrize("i", range(6))
def test_fuzz_context_parallel(orc, i):
    from kimi_delta_attention_13_gb300.context_parallel import prefill_cp

    rng = np.random.default_rng(5000 + i)
    lengths = [int(rng.integers(0, 2500)) for _ in range(int(rng.integers(1, 4)))]
    H = int(rng.integers(1, 4))
    seg_len = int(rng.choice([32, 100, 256, 777]))
    x = synth.make_inputs(lengths, heads=H, dtype="bf16", seed=5000 + i, device=DEV,
                          init_state=bool(rng.random() < 0.5))
    out, fin = prefill_cp(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                          seg_len=seg_len, lengths=lengths)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rf, _ = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu().long(),
                            x["state"])
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final", fin, rf, TOL["bf16"]["state"])
