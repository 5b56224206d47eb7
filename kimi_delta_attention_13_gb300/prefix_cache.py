"""Prefix reuse for KDA serving: resume a request from a stored state checkpoint.

Page "Kimi K3 im Detail: Delta Attention, Attention über Schichten und LatentMoE", section
"Sequenz-Mixing: KDA-Zustand und globale MLA": a reused prefix has to restart from the KDA state
at the same token boundary, and that state is stored only at sparse checkpoints. A request whose
first tokens match a cached sequence therefore:
1. restores the state of the longest checkpoint within the shared prefix (`kda_state_copy`);
2. prefills only the tokens after it, starting from that state (`kda_prefill` with `init_state`).

`CheckpointStore` is a device pool of checkpoint slots with a host-side index. It takes the
checkpoints a prefill emitted (`ckpt_stride`, `ckpts`), and answers "which slot holds the state
after n tokens of sequence `key`". `resume_prefill` restores a batch of requests from their slots in
one `kda_state_copy` and runs one varlen `kda_prefill` over their remaining tokens.

All device work goes through the library's C ABI; this module only keeps the index.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import num_checkpoints, prefill, state_copy


class CheckpointStore:
    """A pool of `n_slots` fp32 states [n_slots, H, d_k, d_v] on `device`, filled round-robin
    (the oldest entry is overwritten when the pool is full), indexed by (key, tokens covered)."""

    def __init__(self, n_slots: int, heads: int, d_k: int = 128, d_v: int = 128, device=None):
        if n_slots < 1:
            raise ValueError("n_slots must be positive")
        self.states = torch.empty(n_slots, heads, d_k, d_v, device=device, dtype=torch.float32)
        self._index: Dict[Tuple[object, int], int] = {}
        self._owner: List[Optional[Tuple[object, int]]] = [None] * n_slots
        self._next = 0

    @property
    def n_slots(self) -> int:
        return self.states.shape[0]

    def _take_slot(self, entry: Tuple[object, int]) -> int:
        slot = self._next
        self._next = (self._next + 1) % self.n_slots
        old = self._owner[slot]
        if old is not None and self._index.get(old) == slot:
            del self._index[old]
        prev = self._index.get(entry)
        if prev is not None:   # the same checkpoint stored again: its older slot is superseded
            self._owner[prev] = None
        self._owner[slot] = entry
        self._index[entry] = slot
        return slot

    def add_checkpoints(self, keys: Sequence[object], ckpts: torch.Tensor, ckpt_stride: int,
                        lengths: Sequence[int], stream=None) -> List[Tuple[object, int, int]]:
        """Store the checkpoints a prefill of sequences `lengths` emitted with `ckpt_stride`
        (`ckpts` as returned by `prefill`, slots ordered by sequence then position), under the
        sequences' `keys`. Returns (key, tokens covered, slot) per stored checkpoint."""
        if len(keys) != len(lengths):
            raise ValueError("one key per sequence")
        if ckpts.shape[0] != num_checkpoints(lengths, ckpt_stride):
            raise ValueError("ckpts does not match lengths and ckpt_stride")
        entries, src = [], []
        pos = 0
        for key, n in zip(keys, lengths):
            for m in range(1, n // ckpt_stride + 1):
                entries.append((key, m * ckpt_stride))
                src.append(pos)
                pos += 1
        if len(entries) > self.n_slots:
            raise ValueError(f"{len(entries)} checkpoints do not fit {self.n_slots} slots")
        dst = [self._take_slot(e) for e in entries]
        if entries:
            dev = self.states.device
            state_copy(self.states, ckpts, torch.tensor(dst, device=dev, dtype=torch.int64),
                       torch.tensor(src, device=dev, dtype=torch.int64), stream=stream)
        return [(k, n, s) for (k, n), s in zip(entries, dst)]

    def lookup(self, key: object, n_tokens: int) -> Tuple[Optional[int], int]:
        """The slot holding the state after the most tokens of `key`, at most `n_tokens`, and that
        token count; (None, 0) if no checkpoint of `key` lies within the first `n_tokens`."""
        best = (None, 0)
        for (k, covered), slot in self._index.items():
            if k == key and covered <= n_tokens and covered > best[1]:
                best = (slot, covered)
        return best


def resume_prefill(store: CheckpointStore, slots: Sequence[Optional[int]], q, k, v, g, beta,
                   cu_seqlens: torch.Tensor, lengths: Sequence[int], *, out=None,
                   final_state=True, out_dtype=torch.float32, stream=None):
    """Prefill a batch of requests from restored states: request i continues from the state in
    `store` slot `slots[i]` (None: from zeros) over its remaining tokens, packed varlen in q, k,
    v, g, beta with `cu_seqlens` / `lengths`. Returns (out, final_state, init_states)."""
    n = len(lengths)
    if len(slots) != n:
        raise ValueError("one slot per request")
    _, H, dk, dv = store.states.shape
    dev = store.states.device
    init = torch.zeros(n, H, dk, dv, device=dev, dtype=torch.float32)
    pairs = [(i, s) for i, s in enumerate(slots) if s is not None]
    if pairs:
        state_copy(init, store.states,
                   torch.tensor([i for i, _ in pairs], device=dev, dtype=torch.int64),
                   torch.tensor([s for _, s in pairs], device=dev, dtype=torch.int64), stream=stream)
    o, f, _ = prefill(q, k, v, g, beta, cu_seqlens, init, out=out, final_state=final_state,
                      lengths=lengths, out_dtype=out_dtype, stream=stream)
    return o, f, init
