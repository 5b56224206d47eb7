"""Prefix reuse through the C ABI: a request that shares a prefix with a cached sequence restores
the checkpoint at the largest stored boundary within that prefix (kda_state_copy) and prefills
only the tokens after it; its outputs and final state equal those of prefilling the whole
sequence (fp64 oracle)."""
import pytest
import torch

import kimi_delta_attention_13_gb300 as kda
import oracle
from kimi_delta_attention_13_gb300 import synth
from kimi_delta_attention_13_gb300.prefix_cache import CheckpointStore, resume_prefill
from parity import TOL, assert_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
KEYS = ("q", "k", "v", "g", "beta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__

    __graft_entry__.build()


def _cat(parts):
    return {key: torch.cat([p[key] for p in parts], 0).contiguous() for key in KEYS}


def _cu(lengths):
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths), 0)
    return cu.to(DEV)


def test_cache_hit_prefill_equals_full_prefill():
    H, base_len, stride = 4, 1024, 256
    base = synth.make_inputs([base_len], heads=H, dtype="bf16", seed=41, device=DEV)
    _, _, ck = kda.prefill(*[base[k] for k in KEYS], ckpt_stride=stride, lengths=[base_len])
    store = CheckpointStore(6, H, device=DEV)   # 4 checkpoints of the base + room
    stored = store.add_checkpoints(["base"], ck, stride, [base_len])
    assert [n for _, n, _ in stored] == [256, 512, 768, 1024]

    # requests: shared prefix length (tokens of the base) and new tokens after it
    prefixes, suffix_lens = [300, 768, 1024, 100], [100, 64, 1, 50]
    suff = synth.make_inputs(suffix_lens, heads=H, dtype="bf16", seed=42, device=DEV)
    offs = [0]
    for n in suffix_lens:
        offs.append(offs[-1] + n)
    suffix = [{key: suff[key][offs[i]:offs[i + 1]] for key in KEYS} for i in range(len(prefixes))]
    base_part = lambda a, b: {key: base[key][a:b] for key in KEYS}  # noqa: E731

    hits = [store.lookup("base", p) for p in prefixes]
    assert [c for _, c in hits] == [256, 768, 1024, 0]
    resume_parts, resume_lens, full_parts, full_lens = [], [], [], []
    for (slot, covered), p, sfx, n in zip(hits, prefixes, suffix, suffix_lens):
        resume_parts += [base_part(covered, p), sfx]
        resume_lens.append(p - covered + n)
        full_parts += [base_part(0, p), sfx]
        full_lens.append(p + n)
    r = _cat(resume_parts)
    out, fin, _ = resume_prefill(store, [s for s, _ in hits], *[r[k] for k in KEYS], _cu(resume_lens),
                                 resume_lens)
    torch.cuda.synchronize()
    assert kda.device_status() == 0

    f = _cat(full_parts)
    ro, rf, _ = oracle.default().prefill(*[f[k] for k in KEYS], _cu(full_lens).cpu(), None)
    # the outputs of the resumed tokens are the last resume_lens[i] outputs of request i
    ref_rows, start = [], 0
    for full_n, res_n in zip(full_lens, resume_lens):
        ref_rows.append(ro[start + full_n - res_n:start + full_n])
        start += full_n
    import numpy as np

    assert_close("out", out, np.concatenate(ref_rows, 0), TOL["bf16"]["out"])
    assert_close("final", fin, rf, TOL["bf16"]["state"])


def test_store_evicts_the_oldest_slot():
    store = CheckpointStore(2, 1, device=DEV)
    ck = torch.zeros(3, 1, 128, 128, device=DEV)
    ck[0] += 1.0
    ck[1] += 2.0
    ck[2] += 3.0
    store.add_checkpoints(["a"], ck[:2], 64, [128])
    store.add_checkpoints(["b"], ck[2:], 64, [64])     # overwrites a's first checkpoint
    torch.cuda.synchronize()
    assert store.lookup("a", 64) == (None, 0)
    slot, covered = store.lookup("a", 1000)
    assert covered == 128 and float(store.states[slot].mean()) == 2.0
    slot, covered = store.lookup("b", 64)
    assert covered == 64 and float(store.states[slot].mean()) == 3.0
