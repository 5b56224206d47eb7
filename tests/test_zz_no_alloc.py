"""kda_prefill_staged_static: the staged prefill with its sequence tables in the library's fixed
device array instead of caller scratch.  It must give kda_prefill_staged's results bit for bit,
stay correct when calls on two streams reuse the array back to back, and refuse (before any CUDA
call) a request whose tables do not fit."""
import ctypes

import numpy as np
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
from kimi_delta_attention_13_gb300 import _lib, build, synth


def test_refuses_tables_larger_than_the_array():
    build.build()
    lib = _lib.load()
    # 2^20 + 1 one-token sequences in chunks of 3 tokens need more than 2^20 table entries
    n = (1 << 20) + 1
    cu = np.arange(n + 1, dtype=np.int32)
    assert lib.kda_prefill_staged_scratch(cu.ctypes.data, n, n, 3) > (1 << 20)
    A = 1 << 20
    args = [A + 16 * i for i in range(5)] + [cu.ctypes.data, n, n, 1, 0, 1, None] + \
        [A + 4096 + 16 * i for i in range(6)] + [A + 2048, A + 8192, 3, None]
    assert lib.kda_prefill_staged_static(*args) == 1   # KDA_ERR_INVALID_ARG


def _host(x):
    return {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}


@pytest.mark.gpu
def test_static_tables_match_caller_scratch():
    dev = torch.device("cuda", 0)
    lengths = [300, 1, 0, 700, 50]
    x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=91, device=dev, init_state=True)
    h, cu = _host(x), x["cu_seqlens"].cpu()
    a, fa, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], cu, x["state"], chunk_tokens=128)
    b, fb, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], cu, x["state"], chunk_tokens=128,
                                  static_tables=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(fa, fb)
    assert kda.device_status() == 0


@pytest.mark.gpu
def test_two_streams_reuse_the_tables_in_order():
    dev = torch.device("cuda", 0)
    runs = []
    for seed, lengths in ((92, [200, 90, 333]), (93, [17, 400, 1, 100])):
        x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=seed, device=dev, init_state=True)
        ref, rf, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"])
        runs.append((x, _host(x), ref, rf))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=dev) for _ in runs]
    outs = []
    for (x, h, _, _), s in zip(runs, streams):   # enqueued back to back on two streams
        outs.append(kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], x["cu_seqlens"].cpu(),
                                       x["state"], chunk_tokens=64, static_tables=True, stream=s))
    torch.cuda.synchronize()
    for (x, _, ref, rf), (o, f, _) in zip(runs, outs):
        # chunk edges cut sequences off their 32-token step grid, which reorders the rounding:
        # compare with kda_prefill within the bf16 bounds
        err_o = float((o - ref.cpu()).abs().max() / ref.cpu().pow(2).mean().sqrt())
        err_f = float((f - rf).abs().max() / rf.pow(2).mean().sqrt())
        assert err_o <= 2e-2 and err_f <= 1e-2, (err_o, err_f)
    assert kda.device_status() == 0
