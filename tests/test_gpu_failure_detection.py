"""Failure detection on the GPU without a fault, and output containment.

1. A bounded device wait that runs out (on a barrier that nothing completes) surfaces as
   KDA_ERR_DEVICE_TIMEOUT through kda_device_status, the read clears it, and the context stays
   usable: a prefill right after it is parity-exact against the oracle.
2. Guard canaries around out, final_state and ckpts stay untouched by every write path (the TMA
   tile store of full 32-token steps, the direct stores of ragged tails, checkpoints, final states).
"""
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
KDA_ERR_DEVICE_TIMEOUT = 5
SENTINEL = 12345.0
GUARD = 1024     # elements of guard on each side (keeps the 16-byte alignment of the views)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def test_expired_device_wait_is_reported_and_context_survives():
    assert kda.device_status() == 0
    kda.diag_device_timeout(2_000_000)          # about 1 ms of SM clock
    torch.cuda.synchronize()
    assert kda.device_status() == KDA_ERR_DEVICE_TIMEOUT
    assert kda.device_status() == 0             # read and cleared
    x = synth.make_inputs([77], heads=2, dtype="bf16", seed=21, device=DEV, init_state=True)
    out, fin, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                              lengths=x["lengths"])
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    ro, rf, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         x["cu_seqlens"].cpu(), x["state"])
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final", fin, rf, TOL["bf16"]["state"])


def _guarded(shape, dtype):
    n = 1
    for d in shape:
        n *= d
    buf = torch.full((n + 2 * GUARD,), SENTINEL, device=DEV, dtype=dtype)
    return buf, buf[GUARD:GUARD + n].view(shape)


def _guards_intact(buf):
    lo, hi = buf[:GUARD], buf[-GUARD:]
    return bool((lo == SENTINEL).all()) and bool((hi == SENTINEL).all())


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("path", ["prefill", "precise", "recurrent"])
def test_writes_stay_inside_their_buffers(path, out_dtype):
    # sequences ending on a full step, on a ragged tail, shorter than a step, and empty
    lengths, H, stride = [128, 100, 5, 0, 64], 3, 64
    x = synth.make_inputs(lengths, heads=H, dtype="bf16", seed=22, device=DEV, init_state=True)
    T, N = sum(lengths), len(lengths)
    n_ck = kda.num_checkpoints(lengths, stride)
    obuf, out = _guarded((T, H, 128), out_dtype)
    fbuf, fin = _guarded((N, H, 128, 128), torch.float32)
    cbuf, ck = _guarded((n_ck, H, 128, 128), torch.float32)
    fn = kda.prefill_recurrent if path == "recurrent" else kda.prefill
    kw = {"precise": True} if path == "precise" else {}
    fn(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"], out=out,
       final_state=fin, ckpts=ck, ckpt_stride=stride, lengths=lengths, out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    for name, b in (("out", obuf), ("final_state", fbuf), ("ckpts", cbuf)):
        assert _guards_intact(b), f"{name}: a write left its buffer"
    assert not bool((out.float() == SENTINEL).any()), "an output row was not written"
