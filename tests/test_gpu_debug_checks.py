"""Device-side bounds checks of the tensor-core prefill.

A library built with -DKDA_DEBUG checks every shared-memory pointer the prefill kernel's accessors
take against its CTA's shared-memory window, and every TMEM address against the allocated columns
and the lanes the executing warp may reach; a failed check skips the access and records
KDA_ERR_DEVICE_BOUNDS (and the check's site) instead of trapping.  Here: the check records a
failure (kda_diag_bounds_check runs it on an out-of-window offset, with no access), and the
debug build runs the small cases, ragged tails and checkpoints included, without a failed check
and within the oracle's bounds, in the default and the precise kernel."""
import ctypes

import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import _lib, build, synth
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def dlib():
    import __graft_entry__

    __graft_entry__.build()
    lib = ctypes.CDLL(build.build(debug=True))
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    yield lib
    torch.cuda.empty_cache()


def _site(lib, run_probe=0):
    site = ctypes.c_int32(-1)
    assert lib.kda_diag_bounds_check(run_probe, ctypes.byref(site), None) == 0
    return site.value


def _status(lib):
    st = ctypes.c_int32(-1)
    assert lib.kda_device_status(ctypes.byref(st), None) == 0
    return st.value


def test_a_failed_check_is_recorded_and_cleared():
    lib = _lib.load()
    assert _site(lib, run_probe=1) == 99           # the probe's site number
    assert kda.device_status() == 7                 # KDA_ERR_DEVICE_BOUNDS
    assert kda.device_status() == 0 and _site(lib) == 0
    # the context is unharmed: a prefill afterwards is exact against the oracle
    x = synth.make_inputs([40], heads=2, dtype="bf16", seed=111, device=DEV)
    out, fin, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"])
    torch.cuda.synchronize()
    ro, rf, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], None, None)
    assert_close("out", out, ro, TOL["bf16"]["out"])


@pytest.mark.parametrize("entry", ["kda_prefill", "kda_prefill_precise"])
@pytest.mark.parametrize("lengths", [[1], [15], [16], [17], [33], [100, 5, 0, 64]])
def test_debug_build_small_cases(dlib, lengths, entry):
    H, stride = 2, 32
    x = synth.make_inputs(lengths, heads=H, dtype="bf16", seed=112 + sum(lengths), device=DEV,
                          init_state=True)
    T, n = sum(lengths), len(lengths)
    out = torch.empty((T, H, 128), device=DEV)
    fin = torch.empty((n, H, 128, 128), device=DEV)
    slots = kda.num_checkpoints(lengths, stride)
    ck = torch.empty((max(slots, 1), H, 128, 128), device=DEV)
    p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    rc = getattr(dlib, entry)(p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]), p(x["cu_seqlens"]), n,
                              T, H, 128, 128, 0, 1, p(x["state"]), p(out), p(fin), stride if slots else 0,
                              p(ck) if slots else None, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert _status(dlib) == 0 and _site(dlib) == 0   # no bounds check failed
    ro, rf, rc_ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"].cpu().long(),
                                           x["state"], ckpt_stride=stride)
    assert_close("out", out, ro, TOL["bf16"]["out"])
    assert_close("final_state", fin, rf, TOL["bf16"]["state"])
    if slots:
        assert_close("ckpts", ck[:slots], rc_, TOL["bf16"]["state"])
