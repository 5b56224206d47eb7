"""The cross-rank context-parallel prefill on CPU: two gloo ranks on 127.0.0.1.

Each rank prefills its own contiguous block of segments, one all-gather shares every segment's
(M, S_loc), and each rank scans and corrects the outputs of its block.  Here the segment prefills
are the fp64 oracle's and the scan a plain fp64 loop, so the assembled outputs and final states
must equal the oracle's prefill of the whole batch up to fp64 rounding: this checks the segment
assignment, the ordering of the gathered slots, the start states handed to each block and the
ownership of every sequence's final state.  (The recurrence is affine in the state, "Kimi K3 im
Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA", which is what makes the split exact.)
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from kimi_delta_attention_13_gb300.context_parallel import (_prefill_cp_ranks, assign_segments,
                                                             gather_segments, segments)

# 13 segments: two ranks own 7 and 6, and the third sequence (330 tokens, 6 segments) crosses the
# boundary; three ranks own 5, 4 and 4, the middle block inside that sequence
LENGTHS, HEADS, SEG_LEN, SEED = [150, 0, 330, 97, 1], 2, 64, 61


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _OracleBackend:
    """The passes' compute on the host: the oracle's prefill and the scan written out."""

    def __init__(self):
        import oracle

        self.orc = oracle.default()

    def prefill(self, q, k, v, g, beta, cu, init):
        o, f, _ = self.orc.prefill(q, k, v, g, beta, cu.long(), init)
        return torch.from_numpy(o), torch.from_numpy(f)

    def scan(self, s_loc, m, seq_seg, s_start):
        fin = []
        for n in range(len(seq_seg) - 1):
            lo, hi = seq_seg[n], seq_seg[n + 1]
            s = s_loc[lo]
            for j in range(lo + 1, hi):
                s_start[j] = s
                s = torch.matmul(m[j], s) + s_loc[j]
            fin.append(s)
        return torch.stack(fin)

    def correct(self, out, u, s_start, cu, skip):
        # out[t, h, :] += u[t, h, :] S_start[seg, h] for the tokens of every segment not skipped
        for j in range(s_start.shape[0]):
            if j in skip:
                continue
            a, b = int(cu[j]), int(cu[j + 1])
            out[a:b] += torch.einsum("thm,hmj->thj", u[a:b], s_start[j])
        return out


def _inputs():
    from kimi_delta_attention_13_gb300 import synth

    x = synth.make_inputs(LENGTHS, heads=HEADS, dtype="bf16", seed=SEED, init_state=True)
    x["state"] = x["state"].double()
    return x


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the gather alone: block sizes differ (5 segments on 2 ranks), slots arrive in order
        owned = assign_segments(5, world)
        mine = torch.tensor([[float(j)] * 3 for j in owned[rank]], dtype=torch.float64)
        got = gather_segments(mine.reshape(len(owned[rank]), 3), owned)
        x = _inputs()
        out, (t0, t1), finals = _prefill_cp_ranks(x["q"], x["k"], x["v"], x["g"], x["beta"], LENGTHS,
                                                  x["state"], SEG_LEN, _OracleBackend())
        results[rank] = (got.numpy(), None if out is None else out.numpy(), t0, t1,
                         {n: f.numpy() for n, f in finals.items()})
    finally:
        dist.destroy_process_group()


def test_assign_segments_covers_each_segment_once():
    for n_seg in (0, 1, 5, 16, 17):
        for world in (1, 2, 3, 8):
            owned = assign_segments(n_seg, world)
            flat = [j for r in owned for j in r]
            assert flat == list(range(n_seg))
            sizes = [len(r) for r in owned]
            assert max(sizes) - min(sizes) <= 1


@pytest.mark.timeout(300)
@pytest.mark.parametrize("world", [2, 3])
def test_ranks_match_the_whole_prefill(world):
    import oracle

    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    # the gathered slots are every segment, in order, on both ranks
    for rank in range(world):
        got = res[rank][0]
        assert np.array_equal(got[:, 0], np.arange(5, dtype=np.float64))
    x = _inputs()
    ro, rf, _ = oracle.default().prefill(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                         x["cu_seqlens"].long(), x["state"])
    bounds, seq_seg = segments(LENGTHS, SEG_LEN)
    owned = assign_segments(len(bounds), world)
    # the case is meant to have, with two ranks, a sequence split across them, and with three, a
    # rank that holds only middle segments of one sequence (no start to skip, no final state)
    if world == 2:
        assert any(seq_seg[n] in owned[0] and seq_seg[n + 1] - 1 in owned[1] for n in range(len(LENGTHS)))
    if world == 3:
        starts, ends = set(seq_seg[:-1]), {j - 1 for j in seq_seg[1:]}
        assert not (set(owned[1]) & starts) and not (set(owned[1]) & ends)
    T = sum(LENGTHS)
    out = np.full((T, HEADS, 128), np.nan)
    seen = {}
    prev_end = 0
    for rank in range(world):
        _, o, t0, t1, fin = res[rank]
        if o is None:
            continue
        assert t0 == prev_end   # the ranks' token blocks tile the batch in rank order
        prev_end = t1
        out[t0:t1] = o
        for n, f in fin.items():
            assert n not in seen
            seen[n] = f
    assert prev_end == T and sorted(seen) == list(range(len(LENGTHS)))
    rms = float(np.sqrt(np.mean(ro ** 2)))
    assert float(np.max(np.abs(out - ro))) <= 1e-9 * rms
    srms = float(np.sqrt(np.mean(rf ** 2)))
    for n, f in seen.items():
        assert float(np.max(np.abs(f - rf[n]))) <= 1e-9 * srms


def test_cp_combine_refuses_a_bad_segment_table():
    # checked on the host before anything reaches the device (no GPU needed to see the refusal)
    import torch

    from kimi_delta_attention_13_gb300.context_parallel import cp_combine

    t = torch.zeros(3, 1, 128, 128)
    for bad in ([1, 3], [0, 2, 1, 3], [0, 4], []):
        with pytest.raises(ValueError, match="seq_seg"):
            cp_combine(t, t, bad, t)
