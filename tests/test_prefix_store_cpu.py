"""Host logic of the prefix-reuse store, on the CPU: which checkpoints a prefill's `ckpts` rows
are, which slots they go to (round-robin, the oldest overwritten), what `lookup` answers, and
which (request, slot) pairs `resume_prefill` restores.  The device copies are recorded instead of
run; the GPU tests check the copies and the resumed prefill against the oracle."""
import pytest
import torch

from kimi_delta_attention_13_gb300 import num_checkpoints, prefix_cache
from kimi_delta_attention_13_gb300.prefix_cache import CheckpointStore, resume_prefill


@pytest.fixture
def copies(monkeypatch):
    log = []

    def fake_state_copy(dst, src, dst_idx=None, src_idx=None, n=None, stream=None):
        log.append((dst, src, dst_idx.tolist(), src_idx.tolist()))

    monkeypatch.setattr(prefix_cache, "state_copy", fake_state_copy)
    return log


def test_checkpoint_rows_and_slots(copies):
    store = CheckpointStore(8, heads=2, d_k=4, d_v=4, device="cpu")
    lengths = [130, 40, 200]          # stride 64: 2, 0 and 3 checkpoints
    assert num_checkpoints(lengths, 64) == 5
    ck = torch.zeros(5, 2, 4, 4)
    stored = store.add_checkpoints(["a", "b", "c"], ck, 64, lengths)
    assert stored == [("a", 64, 0), ("a", 128, 1), ("c", 64, 2), ("c", 128, 3), ("c", 192, 4)]
    (_, _, dst, src), = copies
    assert dst == [0, 1, 2, 3, 4] and src == [0, 1, 2, 3, 4]
    assert store.lookup("a", 130) == (1, 128)
    assert store.lookup("a", 127) == (0, 64)
    assert store.lookup("a", 63) == (None, 0)
    assert store.lookup("b", 10 ** 6) == (None, 0)    # shorter than the stride: nothing stored
    assert store.lookup("c", 10 ** 6) == (4, 192)
    assert store.lookup("z", 10 ** 6) == (None, 0)


def test_round_robin_eviction(copies):
    store = CheckpointStore(3, heads=1, d_k=4, d_v=4, device="cpu")
    store.add_checkpoints(["a"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 0, 1
    stored = store.add_checkpoints(["b"], torch.zeros(2, 1, 4, 4), 32, [70])   # slots 2, 0
    assert [s for _, _, s in stored] == [2, 0]
    assert copies[-1][2] == [2, 0] and copies[-1][3] == [0, 1]
    assert store.lookup("a", 64) == (1, 64)           # a's 32-token checkpoint was overwritten
    assert store.lookup("a", 40) == (None, 0)
    assert store.lookup("b", 64) == (0, 64)
    # the same (key, tokens) stored again takes a new slot; the index points at the newest
    store.add_checkpoints(["a"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 1, 2
    assert store.lookup("a", 64) == (2, 64) and store.lookup("a", 32) == (1, 32)
    assert store.lookup("b", 64) == (0, 64) and store.lookup("b", 32) == (None, 0)


def test_store_errors(copies):
    with pytest.raises(ValueError):
        CheckpointStore(0, heads=1, device="cpu")
    store = CheckpointStore(2, heads=1, d_k=4, d_v=4, device="cpu")
    with pytest.raises(ValueError):
        store.add_checkpoints(["a", "b"], torch.zeros(1, 1, 4, 4), 32, [32])     # keys vs lengths
    with pytest.raises(ValueError):
        store.add_checkpoints(["a"], torch.zeros(1, 1, 4, 4), 32, [64])          # 2 rows expected
    with pytest.raises(ValueError):
        store.add_checkpoints(["a"], torch.zeros(3, 1, 4, 4), 32, [96])          # 3 rows, 2 slots
    assert store.add_checkpoints(["a"], torch.zeros(0, 1, 4, 4), 32, [31]) == []
    assert copies == []                                # nothing to copy, nothing enqueued


def test_resume_restores_only_requests_with_a_slot(copies, monkeypatch):
    store = CheckpointStore(4, heads=1, d_k=4, d_v=4, device="cpu")
    seen = {}

    def fake_prefill(q, k, v, g, beta, cu_seqlens, init, **kw):
        seen["init"], seen["lengths"] = init, kw["lengths"]
        return "out", "final", None

    monkeypatch.setattr(prefix_cache, "prefill", fake_prefill)
    out, fin, init = resume_prefill(store, [3, None, 1], None, None, None, None, None,
                                    torch.tensor([0, 5, 9, 12], dtype=torch.int32), [5, 4, 3])
    assert (out, fin) == ("out", "final") and seen["init"] is init and seen["lengths"] == [5, 4, 3]
    assert init.shape == (3, 1, 4, 4) and not init.any()   # zeros unless restored
    (dst, src, dst_idx, src_idx), = copies
    assert dst is init and src is store.states and dst_idx == [0, 2] and src_idx == [3, 1]
    with pytest.raises(ValueError):
        resume_prefill(store, [None], None, None, None, None, None, None, [5, 4])


def test_checkpoint_stored_again_supersedes_its_older_slot(copies):
    # (a, 32) and (a, 64) stored twice: the first copies (slots 0, 1) are superseded by slots 2, 3;
    # reusing slots 0 and 1 later must not drop the index entries of slots 2 and 3
    store = CheckpointStore(4, heads=1, d_k=4, d_v=4, device="cpu")
    store.add_checkpoints(["a"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 0, 1
    store.add_checkpoints(["a"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 2, 3
    assert store.lookup("a", 32) == (2, 32) and store.lookup("a", 64) == (3, 64)
    store.add_checkpoints(["b"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 0, 1
    assert store.lookup("a", 32) == (2, 32) and store.lookup("a", 64) == (3, 64)
    assert store.lookup("b", 64) == (1, 64)
    store.add_checkpoints(["c"], torch.zeros(2, 1, 4, 4), 32, [64])     # slots 2, 3
    assert store.lookup("a", 64) == (None, 0) and store.lookup("b", 64) == (1, 64)
    assert store.lookup("c", 64) == (3, 64)
