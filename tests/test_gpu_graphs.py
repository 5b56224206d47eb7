"""The library's calls inside CUDA graphs.  A call enqueues only kernel launches on the caller's
stream (no allocation, no host synchronisation), so a captured prefill, decode step or pre-mixer
replays with exactly the eager results, and reads its input buffers anew at every replay."""
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
from kimi_delta_attention_13_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()
    yield
    torch.cuda.empty_cache()


def capture(fn):
    """fn once eagerly on a side stream (first-call set-up), then captured into a graph."""
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(DEV).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


@pytest.mark.parametrize("precise", [False, True])
def test_prefill_graph_replays_bit_identically(precise):
    x = synth.make_inputs([300, 1, 700], heads=4, dtype="bf16", seed=91, device=DEV, init_state=True)
    args = lambda: (x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"])  # noqa: E731
    ref_o, ref_f, ref_c = kda.prefill(*args(), ckpt_stride=128, lengths=x["lengths"], precise=precise)
    out, fin, ck = torch.empty_like(ref_o), torch.empty_like(ref_f), torch.empty_like(ref_c)
    graph = capture(lambda: kda.prefill(*args(), out=out, final_state=fin, ckpt_stride=128, ckpts=ck,
                                        lengths=x["lengths"], precise=precise))
    for t in (out, fin, ck):
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f) and torch.equal(ck, ref_c)
    # new values in the same input buffers: the replay computes with them
    x["v"].mul_(0.5)
    x["state"].mul_(-1.0)
    ref2_o, ref2_f, _ = kda.prefill(*args(), ckpt_stride=128, lengths=x["lengths"], precise=precise)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2_o) and torch.equal(fin, ref2_f)
    assert kda.device_status() == 0


def test_decode_step_graph_as_a_loop():
    N, H = 8, 6
    d = synth.make_decode_inputs(N, heads=H, seed=92, device=DEV)
    state0 = d["state"].clone()
    eager = state0.clone()
    outs = [kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], eager).clone() for _ in range(3)]
    state = state0.clone()
    o = torch.empty(N, H, 128, device=DEV)
    graph = capture(lambda: kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], state, out=o))
    state.copy_(state0)   # undo the eager warm-up step
    for i in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, outs[i]), i
    assert torch.equal(state, eager)
    assert kda.device_status() == 0


def test_premix_graph_with_its_dependent_gates_launch():
    x = synth.make_premix_inputs([200, 57], heads=8, d=128, dtype="bf16", seed=93, device=DEV, hist=True)
    args = (x["xq"], x["xk"], x["xv"], x["a"], x["b"], x["w"], x["cu_seqlens"], x["hist"])
    ref = kda.premix(*args)
    outs = tuple(torch.empty_like(t) for t in ref)
    graph = capture(lambda: kda.premix(*args, out=outs))
    for t in outs:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(outs, ref))
    assert kda.device_status() == 0
