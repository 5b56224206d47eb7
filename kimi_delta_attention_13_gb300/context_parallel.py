"""Context-parallel prefill on one GPU: a sequence split into segments that prefill side by side.

A (sequence, head) chain is serial, so a prefill of few heads keeps few SMs busy (8 heads: 8 of
152).  The recurrence is affine in the state (page "Kimi K3 im Detail", section "Sequenz-Mixing:
KDA-Zustand und globale MLA": per token S_t = A_t S_(t-1) + beta_t k_t v_t^T with
A_t = (I - beta_t k_t k_t^T) diag(exp(g_t))), so over a segment S_end = M S_start + S_loc, and
  1. kda_prefill of every segment as its own sequence, from zeros (a sequence's first segment from
     the sequence's own initial state), gives S_loc;
  2. kda_prefill of every segment with v = 0 from the identity gives M;
  3. kda_cp_combine scans S_start(j + 1) = M(j) S_start(j) + S_loc(j) over each sequence;
  4. kda_prefill of every segment from its true start state gives the outputs and, in each
     sequence's last segment, its final state.
Each of the three prefills runs segments x heads CTAs at once instead of heads, at about three
times a plain prefill's work.  Everything runs in the library's kernels through its C ABI; this
module builds the segment table and moves states between the passes.
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib, _ptr, _require, _stream, prefill, state_copy


def segments(lengths: Sequence[int], seg_len: int) -> Tuple[List[Tuple[int, int]], List[int]]:
    """Token ranges [start, end) of the segments (seg_len tokens, the last of a sequence shorter;
    every sequence at least one, possibly empty) and the per-sequence segment ranges seq_seg."""
    if seg_len < 1:
        raise ValueError("seg_len must be positive")
    bounds, seq_seg, pos = [], [0], 0
    for L in lengths:
        L = int(L)
        if L < 0:
            raise ValueError("negative sequence length")
        starts = range(pos, pos + L, seg_len) if L > 0 else [pos]
        for s in starts:
            bounds.append((s, min(s + seg_len, pos + L)))
        seq_seg.append(len(bounds))
        pos += L
    return bounds, seq_seg


def auto_seg_len(total_tokens: int, heads: int, sms: int) -> int:
    """A segment length for one wave on 7/8 of the SMs: (7 sms / 8) / heads segments per sequence
    of `total_tokens`, rounded up to a multiple of the 32-token chain step.  (With every SM busy
    the prefill's step is about a fifth slower: 19 x 8 segments of 13,824 tokens took as long as
    16 x 8 of 16,384 on one GB300.)"""
    per_seq = max(1, (sms * 7 // 8) // max(1, heads))
    per = -(-int(total_tokens) // per_seq)
    return max(32, -(-per // 32) * 32)


def prefill_cp(q, k, v, g, beta, cu_seqlens=None, init_state=None, *, seg_len: int,
               lengths: Optional[Sequence[int]] = None, out=None, final_state=True, stream=None):
    """Varlen KDA prefill with every sequence cut into segments of `seg_len` tokens that prefill
    in parallel (d_k = d_v = 128).  Arguments as for `prefill` (fp32 outputs; no checkpoints);
    `lengths` avoids a device read of cu_seqlens.  Returns (out, final_state)."""
    lib = _lib.load()
    dev = q.device
    T, H, D = q.shape
    if D != 128 or v.shape[-1] != 128:
        raise ValueError("context-parallel prefill needs d_k = d_v = 128")
    if lengths is None:
        lengths = [T] if cu_seqlens is None else torch.diff(cu_seqlens).tolist()
    N = len(lengths)
    if sum(int(L) for L in lengths) != T:
        raise ValueError("lengths do not add up to the token count")
    if init_state is not None:
        _require(init_state, "init_state", dev, torch.float32, (N, H, D, D))
    if final_state is True:
        final_state = torch.empty((N, H, D, D), device=dev, dtype=torch.float32)
    elif final_state is False:
        final_state = None
    elif final_state is not None:
        _require(final_state, "final_state", dev, torch.float32, (N, H, D, D))
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        bounds, seq_seg = segments(lengths, seg_len)
        n_seg = len(bounds)
        cu_seg = torch.tensor([b for b, _ in bounds] + [T], dtype=torch.int32, device=dev)
        first = torch.tensor(seq_seg[:-1], dtype=torch.int64, device=dev)
        last = torch.tensor([i - 1 for i in seq_seg[1:]], dtype=torch.int64, device=dev)
        seqs = torch.arange(N, device=dev)
        # 1. every segment from zeros; a sequence's first segment from its own initial state
        init_seg = torch.zeros((n_seg, H, D, D), device=dev, dtype=torch.float32)
        if init_state is not None and N > 0:
            state_copy(init_seg, init_state, first, seqs, stream=s)
        out, s_loc, _ = prefill(q, k, v, g, beta, cu_seg, init_seg, out=out, final_state=True, stream=s)
        if n_seg == N:   # no sequence was split: the pass above is the whole prefill
            if final_state is not None and N > 0:
                state_copy(final_state, s_loc, stream=s)
            return out, final_state
        # 2. every segment with v = 0 from the identity: the segment maps M (outputs unused)
        eye = torch.eye(D, device=dev, dtype=torch.float32).expand(n_seg, H, D, D).contiguous()
        scratch = torch.empty_like(out)
        _, m, _ = prefill(q, k, torch.zeros_like(v), g, beta, cu_seg, eye, out=scratch,
                          final_state=True, stream=s)
        del eye, scratch
        # 3. each segment's true start state (a first segment keeps its sequence's initial state)
        s_start = init_seg
        seq_seg_t = torch.tensor(seq_seg, dtype=torch.int32, device=dev)
        rc = lib.kda_cp_combine(_ptr(s_loc), _ptr(m), _ptr(seq_seg_t), N, H, D, _ptr(s_start),
                                None, _stream(dev, s))
        _lib.check(rc, "kda_cp_combine")
        del m
        # 4. every segment from its true start: the outputs, and the sequences' final states
        out, seg_final, _ = prefill(q, k, v, g, beta, cu_seg, s_start, out=out, final_state=s_loc,
                                    stream=s)
        if final_state is not None and N > 0:
            state_copy(final_state, seg_final, seqs, last, stream=s)
        return out, final_state
