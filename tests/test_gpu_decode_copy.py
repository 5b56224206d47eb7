"""kda_decode and kda_state_copy on the GPU against the fp64 oracle / exact expectations."""
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


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def check_decode(orc, d, dtype):
    S0 = d["state"].clone()
    out = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    torch.cuda.synchronize()
    ro, rs = orc.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], S0)
    e = (assert_close("out", out, ro, TOL[dtype]["out"]),
         assert_close("state", d["state"], rs, TOL[dtype]["state"]))
    return e


@pytest.mark.parametrize("n,dtype", [(1, "bf16"), (5, "bf16"), (7, "f32")])
def test_decode_small(orc, n, dtype):
    d = synth.make_inputs([1] * n, heads=3, dtype=dtype, seed=30 + n, device=DEV, init_state=True)
    check_decode(orc, d, dtype)


@pytest.mark.parametrize("dk,dv", [(64, 32), (1, 4), (128, 4), (100, 68)])
def test_decode_other_head_sizes(orc, dk, dv):
    d = synth.make_inputs([1] * 4, heads=2, d_k=dk, d_v=dv, dtype="f32", seed=dk * dv, device=DEV,
                          init_state=True)
    check_decode(orc, d, "f32")


def test_decode_bf16_outputs(orc):
    d = synth.make_inputs([1] * 9, heads=3, dtype="bf16", seed=35, device=DEV, init_state=True)
    S0 = d["state"].clone()
    out = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ro, rs = orc.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], S0)
    import numpy as np

    g = out.double().cpu().numpy()
    rms = float(np.sqrt(np.mean(ro ** 2)))
    assert out.dtype == torch.bfloat16
    assert np.all(np.abs(g - ro) <= 2e-2 * rms + 2.0 ** -8 * np.abs(ro))


def test_decode_zero_sequences():
    d = synth.make_inputs([], heads=2, dtype="bf16", seed=1, device=DEV, init_state=True)
    out = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    torch.cuda.synchronize()
    assert out.shape == (0, 2, 128) and out.dtype == torch.float32


def test_decode_continues_prefill(orc):
    """decode of token t from the state after t-1 tokens equals row t of a prefill."""
    x = synth.make_inputs([129], heads=2, dtype="bf16", seed=33, device=DEV, init_state=True)
    t = 128
    pre = {k: x[k][:t] for k in ("q", "k", "v", "g", "beta")}
    _, S, _ = kda.prefill(**pre, init_state=x["state"])
    one = {k: x[k][t:t + 1] for k in ("q", "k", "v", "g", "beta")}
    o = kda.decode(**one, state=S)
    torch.cuda.synchronize()
    ro, rf, _ = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    assert_close("out[t]", o[0], ro[t], TOL["bf16"]["out"])
    assert_close("state", S, rf, TOL["bf16"]["state"])


def test_decode_workload_N256(orc):
    w = synth.workloads()[3]
    d = synth.make_workload_inputs(w, DEV)
    e = check_decode(orc, d, "bf16")
    print("decode N256", e)


def test_state_copy_gather_scatter():
    H, dk, dv = 3, 128, 128
    src = torch.randn(6, H, dk, dv, device=DEV)
    dst = torch.zeros(5, H, dk, dv, device=DEV)
    src_idx = torch.tensor([4, 0, 2], device=DEV)
    dst_idx = torch.tensor([1, 3, 0], device=DEV)
    kda.state_copy(dst, src, dst_idx, src_idx)
    torch.cuda.synchronize()
    expect = torch.zeros_like(dst)
    expect[dst_idx] = src[src_idx]
    assert torch.equal(dst, expect)
    assert kda.device_status() == 0


def test_state_copy_count_is_checked_against_the_indices():
    src = torch.randn(4, 2, 128, 128, device=DEV)
    dst = torch.zeros_like(src)
    idx = torch.tensor([2, 0], device=DEV)
    with pytest.raises(ValueError):
        kda.state_copy(dst, src, idx, idx, n=3)   # 3 entries read from 2-entry index arrays
    torch.cuda.synchronize()
    assert not dst.any()
    kda.state_copy(dst, src, idx, idx, n=1)
    torch.cuda.synchronize()
    assert torch.equal(dst[2], src[2]) and not dst[0].any()


def test_state_copy_identity_and_odd_unit():
    src = torch.randn(3, 1, 3, 5, device=DEV)   # 15 floats per slot: scalar path
    dst = torch.zeros(3, 1, 3, 5, device=DEV)
    kda.state_copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)


def test_state_copy_out_of_range_index_is_reported():
    src = torch.randn(2, 2, 128, 128, device=DEV)
    dst = torch.zeros(2, 2, 128, 128, device=DEV)
    kda.state_copy(dst, src, torch.tensor([0, 7], device=DEV), torch.tensor([1, 0], device=DEV))
    assert kda.device_status() == 6          # KDA_ERR_INDEX_RANGE, sticky until read
    assert kda.device_status() == 0          # cleared by the read
    assert torch.equal(dst[0], src[1])       # the in-range copy happened
    assert torch.count_nonzero(dst[1]) == 0  # the bad one was skipped


def test_checkpoint_restore_resumes(orc):
    """Restore a checkpoint with kda_state_copy and resume: equals the uninterrupted run."""
    x = synth.make_inputs([512], heads=2, dtype="bf16", seed=34, device=DEV, init_state=True)
    _, _, ck = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], init_state=x["state"],
                           ckpt_stride=128, lengths=[512])
    slot = torch.zeros(1, 2, 128, 128, device=DEV)
    kda.state_copy(slot, ck, torch.tensor([0], device=DEV), torch.tensor([1], device=DEV))  # after 256
    rest = {k: x[k][256:].contiguous() for k in ("q", "k", "v", "g", "beta")}
    o2, s2, _ = kda.prefill(**rest, init_state=slot)
    torch.cuda.synchronize()
    ro, rf, _ = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["state"])
    assert_close("out", o2, ro[256:], TOL["bf16"]["out"])
    assert_close("final", s2, rf, TOL["bf16"]["state"])
