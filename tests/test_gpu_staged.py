"""kda_prefill_staged: prefill from pinned host memory with chunked, overlapped copies.  A single
sequence cut at multiples of 32 tokens must give kda_prefill's results bit for bit (the state
passes between chunks in fp32 exactly as between steps); varlen batches with chunks that cut
through sequences must match the fp64 oracle (bf16 bounds)."""
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    yield
    torch.cuda.empty_cache()


def host(x):
    return {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}


def test_single_sequence_is_bit_identical():
    x = synth.make_inputs([2048], heads=4, dtype="bf16", seed=81, device=DEV, init_state=True)
    ref_o, ref_f, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    h = host(x)
    out, fin, bufs = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"],
                                        chunk_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o.cpu()) and torch.equal(fin, ref_f)
    # buffers and outputs reused by a second call, with a ragged last chunk
    out2, fin2, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"],
                                       chunk_tokens=704, buffers=bufs, h_out=out, final_state=fin)
    torch.cuda.synchronize()
    assert torch.equal(out2, ref_o.cpu()) and torch.equal(fin2, ref_f)


@pytest.mark.parametrize("lengths,chunk,out_dtype", [
    ([300, 1, 0, 700, 50], 128, torch.float32),
    ([300, 1, 0, 700, 50], 100, torch.float32),     # chunks not aligned to the 32-token step
    ([64, 64, 64], 64, torch.bfloat16),
])
def test_varlen_against_oracle(lengths, chunk, out_dtype):
    x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=82 + chunk, device=DEV, init_state=True)
    h = host(x)
    out, fin, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], x["cu_seqlens"].cpu(),
                                     x["state"], chunk_tokens=chunk, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rf, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         x["cu_seqlens"].cpu().long(), x["state"])
    tol_out = TOL["bf16"]["out"] if out_dtype == torch.float32 else 4e-2
    assert_close("out", out, ro, tol_out)
    assert_close("final_state", fin, rf, TOL["bf16"]["state"])


def test_edge_cases():
    orc = oracle.default()
    # empty leading and trailing sequences, one chunk larger than all tokens
    lengths = [0, 37, 0, 90, 0]
    x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=85, device=DEV, init_state=True)
    h = host(x)
    out, fin, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], x["cu_seqlens"].cpu(),
                                     x["state"], chunk_tokens=4096)
    torch.cuda.synchronize()
    ro, rf, _ = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu().long(), x["state"])
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final_state", fin, rf, TOL["bf16"]["state"])
    assert torch.equal(fin[0], x["state"][0]) and torch.equal(fin[4], x["state"][4])   # empty: init kept
    # no tokens at all: the final states are the initial ones
    e = synth.make_inputs([0, 0], heads=2, dtype="bf16", seed=86, device=DEV, init_state=True)
    he = host(e)
    out, fin, _ = kda.prefill_staged(he["q"], he["k"], he["v"], he["g"], he["beta"], e["cu_seqlens"].cpu(),
                                     e["state"], chunk_tokens=64)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(fin, e["state"])
    assert kda.device_status() == 0


def test_tail_split_and_pageable_output():
    # 1000 tokens in chunks of 512: the last 488 are cut into 256 + 128 + 104; outputs are
    # downloaded by SM stores into the pinned buffer, and by copies into a pageable one.
    x = synth.make_inputs([1000], heads=3, dtype="bf16", seed=87, device=DEV, init_state=True)
    ref_o, ref_f, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    h = host(x)
    out, fin, bufs = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"],
                                        chunk_tokens=512)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o.cpu()) and torch.equal(fin, ref_f)

    lib = kda._lib.load()
    pageable = torch.full((1000, 3, 128), float("nan"))
    assert not pageable.is_pinned()
    fin2 = torch.empty_like(ref_f)
    rc = lib.kda_prefill_staged(
        kda._ptr(h["q"]), kda._ptr(h["k"]), kda._ptr(h["v"]), kda._ptr(h["g"]), kda._ptr(h["beta"]),
        None, 1, 1000, 3, kda._DTYPES[torch.bfloat16], kda._DTYPES[torch.float32], kda._ptr(x["state"]),
        *[kda._ptr(bufs[k]) for k in ("q", "k", "v", "g", "beta", "out")], kda._ptr(pageable),
        kda._ptr(fin2), None, 0, 512, kda._stream(DEV, None))
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(pageable, ref_o.cpu()) and torch.equal(fin2, ref_f)
    assert kda.device_status() == 0


def test_reused_buffers_must_hold_the_tokens():
    short = synth.make_inputs([64], heads=2, dtype="bf16", seed=88, device=DEV)
    hs = host(short)
    _, _, bufs = kda.prefill_staged(hs["q"], hs["k"], hs["v"], hs["g"], hs["beta"], chunk_tokens=32)
    x = synth.make_inputs([96], heads=2, dtype="bf16", seed=89, device=DEV)
    h = host(x)
    with pytest.raises(ValueError):
        kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], chunk_tokens=32, buffers=bufs)
    torch.cuda.synchronize()
    assert kda.device_status() == 0


def test_unaligned_chunk_size_is_refused_before_any_work():
    # H = 3 bf16 heads: chunks of 100 tokens would start the second chunk's beta rows at byte
    # 600, off the 16-byte grid every prefill pointer keeps; the call refuses it up front
    x = synth.make_inputs([250], heads=3, dtype="bf16", seed=90, device=DEV, init_state=True)
    h = host(x)
    fin = torch.full((1, 3, 128, 128), 7.0, device=DEV)
    with pytest.raises(kda.KDAError, match="INVALID_ARG"):
        kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"], chunk_tokens=100,
                           final_state=fin)
    torch.cuda.synchronize()
    assert bool((fin == 7.0).all())   # nothing was enqueued
    # chunks of 96 tokens x 3 heads keep beta aligned: same call, against the oracle
    out, fin, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"], chunk_tokens=96)
    torch.cuda.synchronize()
    ro, rf, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final_state", fin, rf, TOL["bf16"]["state"])
    assert kda.device_status() == 0


def staged_handles() -> int:
    import ctypes

    from kimi_delta_attention_13_gb300 import _lib

    n = ctypes.c_int64(-1)
    assert _lib.load().kda_diag_staged_handles(ctypes.byref(n)) == 0
    return n.value


def test_repeated_calls_reuse_the_device_streams():
    # the staged call keeps two streams and four events per device after its first call; many
    # calls in a row (and from a second stream) stay exact against one kda_prefill
    x = synth.make_inputs([640], heads=2, dtype="bf16", seed=91, device=DEV, init_state=True)
    ref_o, ref_f, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    h = host(x)
    bufs = None
    s2 = torch.cuda.Stream(device=DEV)
    created = []
    for i in range(20):
        out, fin, bufs = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], None, x["state"],
                                            chunk_tokens=128, buffers=bufs, stream=s2 if i % 2 else None)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o.cpu()) and torch.equal(fin, ref_f)
        created.append(staged_handles())
    # the first call on the device may create the streams and events; no later call creates any
    assert len(set(created)) == 1, created
    assert kda.device_status() == 0
