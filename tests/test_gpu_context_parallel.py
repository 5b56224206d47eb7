"""Context-parallel prefill on the GPU against the fp64 oracle's plain (token by token) prefill:
segments prefilled side by side, joined by kda_cp_combine's scan and kda_cp_correct's output
correction, must give the outputs and final states of the whole sequences (bf16 inputs: 2e-2 x RMS
on outputs, 1e-2 on states)."""
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from kimi_delta_attention_13_gb300.context_parallel import prefill_cp
from parity import TOL, assert_close, head_slice

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


def check(orc, lengths, heads, seg_len, init, seed, oracle_heads=None, decay_scale=1.0):
    x = synth.make_inputs(lengths, heads=heads, dtype="bf16", seed=seed, device=DEV, init_state=init,
                          decay_scale=decay_scale)
    out, fin = prefill_cp(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                          seg_len=seg_len, lengths=lengths)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    hs = list(range(heads)) if oracle_heads is None else oracle_heads
    c = head_slice(x, hs)
    init_c = None if x["state"] is None else x["state"][:, hs].cpu()
    ro, rf, _ = orc.prefill(c["q"], c["k"], c["v"], c["g"], c["beta"], x["cu_seqlens"].cpu().long(), init_c)
    idx = torch.tensor(hs, device=DEV)
    assert_close("out", out.index_select(1, idx), ro, TOL["bf16"]["out"])
    assert_close("final_state", fin.index_select(1, idx), rf, TOL["bf16"]["state"])
    return x, out, fin


@pytest.mark.parametrize("lengths,heads,seg_len,init", [
    ([300, 5, 700], 2, 128, True),      # ragged segments, a sequence shorter than a segment
    ([1000], 3, 64, False),             # many segments
    ([0, 257, 0, 64], 2, 64, True),     # empty sequences, a sequence of exactly one segment
    ([4096], 2, 1000, True),            # segment length not a multiple of the tile
])
def test_cp_matches_oracle(orc, lengths, heads, seg_len, init):
    check(orc, lengths, heads, seg_len, init, seed=sum(lengths) + seg_len)


def test_cp_without_a_split_is_the_plain_prefill(orc):
    x, out, fin = check(orc, [200, 31], 2, 4096, True, seed=71)
    o2, f2, _ = kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"])
    torch.cuda.synchronize()
    assert torch.equal(out, o2) and torch.equal(fin, f2)


def test_cp_long_sequence(orc):
    # 65,536 tokens of 4 heads in 8 segments of 8,192: 32 + 32 CTAs instead of 4
    check(orc, [65536], 4, 8192, True, seed=72)


def test_cp_edge_cases(orc):
    # a single-token sequence next to a long one, and a batch without tokens
    check(orc, [1, 600], 2, 128, True, seed=73)
    e = synth.make_inputs([0, 0], heads=2, dtype="bf16", seed=74, device=DEV, init_state=True)
    out, fin = prefill_cp(e["q"], e["k"], e["v"], e["g"], e["beta"], e["cu_seqlens"], e["state"],
                          seg_len=64, lengths=[0, 0])
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(fin, e["state"])


def test_cp_bench_configuration(orc):
    # the configuration of the benchmark's context-parallel figure: one sequence of 262,144 tokens,
    # 8 heads, the benchmark's seed and segment length (16 segments of 16,384 on 152 SMs); the
    # oracle checks two heads
    from kimi_delta_attention_13_gb300.context_parallel import auto_seg_len

    T, H = 262144, 8
    seg = auto_seg_len(T, H, torch.cuda.get_device_properties(DEV).multi_processor_count)
    check(orc, [T], H, seg, False, seed=9, oracle_heads=[2, 5])


def test_cp_slow_decay(orc):
    # g x 0.01: each segment's map M is far from zero, so the scan composes states that carry
    # across segments (with the workloads' fast decay every M is ~0)
    check(orc, [65536], 4, 8192, True, seed=75, decay_scale=0.01)


def test_cp_distributed_single_rank_equals_one_gpu(orc):
    # the cross-rank call in a group of one (NCCL on this GPU): the same segments, scan and passes
    # as the one-GPU call, so the results are bit-identical
    import socket

    import torch.distributed as dist

    from kimi_delta_attention_13_gb300.context_parallel import prefill_cp_distributed

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=DEV)
    try:
        lengths = [700, 0, 300]
        x = synth.make_inputs(lengths, heads=2, dtype="bf16", seed=76, device=DEV, init_state=True)
        out1, fin1 = prefill_cp(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                                seg_len=128, lengths=lengths)
        out2, (t0, t1), finals = prefill_cp_distributed(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                        x["state"], seg_len=128, lengths=lengths)
        torch.cuda.synchronize()
        assert (t0, t1) == (0, sum(lengths)) and sorted(finals) == [0, 1, 2]
        assert torch.equal(out1, out2)
        for n, f in finals.items():
            assert torch.equal(f, fin1[n])
        assert kda.device_status() == 0
    finally:
        dist.destroy_process_group()


def test_cp_combine_scan_against_fp64():
    # the scan alone on random segment maps: S_start(j + 1) = M(j) S_start(j) + S_loc(j) over each
    # sequence's segments, checked in fp64 on the host; sequences of 0, 1, 2 and 19 segments, and
    # maps of norm about 1 so that every step carries the state forward
    from kimi_delta_attention_13_gb300.context_parallel import cp_combine

    H, D = 3, 128
    seq_seg = [0, 1, 1, 3, 22]
    n_seg = seq_seg[-1]
    gen = torch.Generator().manual_seed(83)
    s_loc = torch.randn(n_seg, H, D, D, generator=gen)
    m = torch.randn(n_seg, H, D, D, generator=gen) / D ** 0.5
    sentinel = 7.25
    s_start = torch.full((n_seg, H, D, D), sentinel)
    fin = torch.full((len(seq_seg) - 1, H, D, D), sentinel)
    d_start, d_fin = s_start.to(DEV), fin.to(DEV)
    cp_combine(s_loc.to(DEV), m.to(DEV), seq_seg, d_start, d_fin)
    torch.cuda.synchronize()
    got_start, got_fin = d_start.cpu(), d_fin.cpu()
    for n in range(len(seq_seg) - 1):
        lo, hi = seq_seg[n], seq_seg[n + 1]
        if hi == lo:
            assert torch.all(got_fin[n] == sentinel)   # no segment: nothing written
            continue
        assert torch.all(got_start[lo] == sentinel)    # a first segment keeps its own start
        s = s_loc[lo].double()
        for j in range(lo + 1, hi):
            err = (got_start[j].double() - s).abs().max() / s.pow(2).mean().sqrt()
            assert err < 1e-4, (n, j, float(err))
            s = m[j].double() @ s + s_loc[j].double()
        err = (got_fin[n].double() - s).abs().max() / s.pow(2).mean().sqrt()
        assert err < 1e-4, (n, float(err))


@pytest.mark.parametrize("bounds,H,skip", [
    ([0, 300, 300, 333, 589, 845, 1130], 3, [0, 3]),   # empty, two exact tiles, ends at the last token
    ([0, 5, 37], 1, []),                               # less than one tile in all
    ([0, 100, 300], 70, [0]),                          # many heads
    ([0, 1, 2, 3, 130], 2, [1]),                       # one-token segments
])
def test_cp_correct_against_fp64(bounds, H, skip):
    """kda_cp_correct alone: out[t] += S_start(seg)^T u_t over ragged segments, with the skipped
    segments left bit for bit.  tf32 operands bound the error of the added term per element by
    (2^-10 + 2^-11) sum_m |u_m| |S_mj| (u truncated, S rounded to nearest); the test allows 2^-9."""
    from kimi_delta_attention_13_gb300.context_parallel import cp_correct

    gen = torch.Generator().manual_seed(71 + H)
    D = 128
    T, n_seg = bounds[-1], len(bounds) - 1
    u = torch.randn(T, H, D, generator=gen)
    out0 = torch.randn(T, H, D, generator=gen)
    s_start = 0.1 * torch.randn(n_seg, H, D, D, generator=gen)
    ref, bound = out0.double().clone(), torch.zeros(T, H, D, dtype=torch.float64)
    for j in range(n_seg):
        a, b = bounds[j], bounds[j + 1]
        if j in skip:
            continue
        ref[a:b] += torch.einsum("thm,hmj->thj", u[a:b].double(), s_start[j].double())
        bound[a:b] = 2.0 ** -9 * torch.einsum("thm,hmj->thj", u[a:b].abs().double(), s_start[j].abs().double())
    out = out0.to(DEV)
    cp_correct(out, u.to(DEV), s_start.to(DEV), torch.tensor(bounds, dtype=torch.int32, device=DEV), skip)
    torch.cuda.synchronize()
    assert kda.device_status() == 0
    got = out.cpu()
    for j in skip:   # left as they were, bit for bit
        a, b = bounds[j], bounds[j + 1]
        assert torch.equal(got[a:b], out0[a:b])
    err = (got.double() - ref).abs()
    assert torch.all(err <= bound + 1e-6 * ref.abs()), float((err - bound).max())
