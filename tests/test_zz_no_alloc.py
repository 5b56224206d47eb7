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


_REFUSAL = r"""
import numpy as np
from kimi_delta_attention_13_gb300 import _lib
lib = _lib.load()
# 2^20 + 1 one-token sequences in chunks of 3 tokens need more than 2^20 table entries
n = (1 << 20) + 1
cu = np.arange(n + 1, dtype=np.int32)
assert lib.kda_prefill_staged_scratch(cu.ctypes.data, n, n, 3) > (1 << 20)
A = 1 << 20   # made-up addresses: the size check must refuse the call before any CUDA call
args = [A + 16 * i for i in range(5)] + [cu.ctypes.data, n, n, 1, 0, 1, None] + \
    [A + 4096 + 16 * i for i in range(6)] + [A + 2048, A + 8192, 3, None]
print("rc", lib.kda_prefill_staged_static(*args))
"""


def test_refuses_tables_larger_than_the_array():
    import os
    import subprocess
    import sys

    build.build()
    # in a process that sees no GPU, so that the made-up addresses can reach no device even if
    # the check before the CUDA calls were lost
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _REFUSAL], cwd=root, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "rc 1" in r.stdout   # KDA_ERR_INVALID_ARG


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
    """Call 1 (many short sequences, 64 chunks) is still running when call 2, on another stream and
    with other sequence tables, is enqueued: without the wait on call 1's last prefill, call 2's
    table upload would overwrite entries call 1's later chunks still read.  Each call must equal
    the caller-scratch call bit for bit (the same chunks, so the same arithmetic)."""
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(94)
    len1 = torch.randint(1, 400, (80,), generator=g).tolist()
    len2 = torch.randint(1, 300, (40,), generator=g).tolist()
    runs = []
    for seed, lengths in ((95, len1), (96, len2)):
        x = synth.make_inputs(lengths, heads=4, dtype="bf16", seed=seed, device=dev, init_state=True)
        h, cu = _host(x), x["cu_seqlens"].cpu()
        ref, rf, _ = kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], cu, x["state"],
                                        chunk_tokens=256)
        torch.cuda.synchronize()   # the downloads into the host buffer are asynchronous
        runs.append((x, h, cu, ref.clone(), rf.clone()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(device=dev) for _ in runs]
    outs = []
    for (x, h, cu, _, _), s in zip(runs, streams):   # enqueued back to back on two streams
        outs.append(kda.prefill_staged(h["q"], h["k"], h["v"], h["g"], h["beta"], cu, x["state"],
                                       chunk_tokens=256, static_tables=True, stream=s))
    torch.cuda.synchronize()
    for (_, _, _, ref, rf), (o, f, _) in zip(runs, outs):
        assert torch.equal(o, ref) and torch.equal(f, rf)
    assert kda.device_status() == 0
