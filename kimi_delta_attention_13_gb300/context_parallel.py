"""Context-parallel prefill on one GPU: a sequence split into segments that prefill side by side.

A (sequence, head) chain is serial, so a prefill of few heads keeps few SMs busy (8 heads: 8 of
152).  The recurrence is affine in the state (page "Kimi K3 im Detail", section "Sequenz-Mixing:
KDA-Zustand und globale MLA": per token S_t = A_t S_(t-1) + beta_t k_t v_t^T with
A_t = (I - beta_t k_t k_t^T) diag(exp(g_t))), so within a segment S_t = P_t S_start + S_loc,t with
P_t = A_t ... A_1, and
  1. kda_prefill of every segment as its own sequence, from zeros (a sequence's first segment from
     the sequence's own initial state), gives S_loc and the outputs o_loc;
  2. kda_prefill of every segment with v = 0 from the identity gives M = P_L and the outputs
     u_t = P_t^T q_t;
  3. kda_cp_combine scans S_start(j + 1) = M(j) S_start(j) + S_loc(j) over each sequence, and
     gives each sequence's final state;
  4. kda_cp_correct adds S_start^T u_t to o_loc,t in every segment that does not start its
     sequence: o_t = S_t^T q_t = o_loc,t + S_start^T u_t.
Each of the two prefills runs segments x heads CTAs at once instead of heads, at about twice a
plain prefill's work.  Everything runs in the library's kernels through its C ABI; this module
builds the segment tables and moves states between the passes.
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


def cp_combine(s_loc, m, seq_seg, s_start, final_state=None, stream=None):
    """The segment scan (kda_cp_combine): for every sequence n and segment j of
    [seq_seg[n], seq_seg[n + 1]), S_start(j + 1) = M(j) S_start(j) + S_loc(j), starting from
    S_loc of the sequence's first segment.  s_loc, m, s_start: fp32 [n_seg, H, 128, 128] on one
    device; seq_seg: n_seqs + 1 segment indices, a host list or an int32 tensor on the device;
    final_state: fp32 [n_seqs, H, 128, 128] or None.  s_start of each sequence's first segment is
    left as it is."""
    dev = s_loc.device
    n_seg, H, D = s_loc.shape[0], s_loc.shape[1], s_loc.shape[2]
    if not isinstance(seq_seg, torch.Tensor):
        seq_seg = [int(v) for v in seq_seg]
        if not seq_seg or seq_seg[0] != 0 or seq_seg[-1] > n_seg or any(
                b < a for a, b in zip(seq_seg, seq_seg[1:])):
            raise ValueError(f"seq_seg must rise from 0 to at most {n_seg} segments")
    for name, t in (("s_loc", s_loc), ("m", m), ("s_start", s_start)):
        _require(t, name, dev, torch.float32, (n_seg, H, D, D))
    if isinstance(seq_seg, torch.Tensor):
        # a device table is taken as it is (its values are not read back to the host), like
        # cu_seqlens: non-decreasing, from 0 to at most n_seg
        _require(seq_seg, "seq_seg", dev, torch.int32)
        if seq_seg.dim() != 1 or seq_seg.numel() < 1:
            raise ValueError("seq_seg must be one-dimensional and non-empty")
    if final_state is not None:
        _require(final_state, "final_state", dev, torch.float32, (len(seq_seg) - 1, H, D, D))
    lib = _lib.load()
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        seq_seg_t = seq_seg if isinstance(seq_seg, torch.Tensor) else \
            torch.tensor(seq_seg, dtype=torch.int32, device=dev)
        rc = lib.kda_cp_combine(_ptr(s_loc), _ptr(m), _ptr(seq_seg_t), len(seq_seg) - 1, H, D,
                                _ptr(s_start), _ptr(final_state) if final_state is not None else None,
                                _stream(dev, s))
    _lib.check(rc, "kda_cp_combine")
    return s_start


def cp_correct(out, u, s_start, cu_seg, skip_seg, stream=None):
    """The output correction (kda_cp_correct): out[t] += S_start(seg)^T u_t for the tokens of every
    segment seg not in skip_seg.  out, u: fp32 [T, H, 128] on one device; s_start: fp32
    [n_seg, H, 128, 128]; cu_seg: int32 [n_seg + 1] token offsets on the device; skip_seg: the
    segments left as they are, an increasing host list or int32 device tensor.  Returns out."""
    dev = out.device
    T, H, D = out.shape
    n_seg = s_start.shape[0]
    _require(out, "out", dev, torch.float32, (T, H, D))
    _require(u, "u", dev, torch.float32, (T, H, D))
    _require(s_start, "s_start", dev, torch.float32, (n_seg, H, D, D))
    _require(cu_seg, "cu_seg", dev, torch.int32, (n_seg + 1,))
    lib = _lib.load()
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.stream(s):
        if not isinstance(skip_seg, torch.Tensor):
            skip = [int(j) for j in skip_seg]
            if any(b <= a for a, b in zip(skip, skip[1:])):
                raise ValueError("skip_seg must be increasing")
            skip_seg = torch.tensor(skip, dtype=torch.int32, device=dev)
        else:
            _require(skip_seg, "skip_seg", dev, torch.int32)
        n_skip = int(skip_seg.numel())
        rc = lib.kda_cp_correct(_ptr(u), _ptr(s_start), _ptr(cu_seg), n_seg,
                                _ptr(skip_seg) if n_skip else None, n_skip, T, H, D, _ptr(out),
                                _stream(dev, s))
    _lib.check(rc, "kda_cp_correct")
    return out


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
        # 2. every segment with v = 0 from the identity: the segment maps M and the outputs u
        eye = torch.eye(D, device=dev, dtype=torch.float32).expand(n_seg, H, D, D).contiguous()
        u = torch.empty((T, H, D), device=dev, dtype=torch.float32)
        _, m, _ = prefill(q, k, torch.zeros_like(v), g, beta, cu_seg, eye, out=u, final_state=True,
                          stream=s)
        del eye
        # 3. each segment's true start state (a first segment keeps its sequence's initial state)
        # and each sequence's final state
        s_start = init_seg
        cp_combine(s_loc, m, seq_seg, s_start, final_state=final_state, stream=s)
        del m
        # 4. the outputs of every segment that does not start its sequence
        cp_correct(out, u, s_start, cu_seg, seq_seg[:-1], stream=s)
        return out, final_state


# --------------------------------------------------------------------------------------------
# Across ranks: each rank owns a contiguous block of the segments.  Passes 1 and 2 run on a
# rank's own segments; one all-gather hands every rank every segment's (M, S_loc); each rank
# runs the (cheap) scan over all segments and the output correction on its own.  The only data
# crossing ranks is that exchange: 2 x H x d x d fp32 per segment.


def assign_segments(n_seg: int, world_size: int) -> List[range]:
    """Contiguous, balanced blocks of segment indices, one per rank (rank r owns owned[r])."""
    if world_size < 1:
        raise ValueError("world_size must be positive")
    base, extra = divmod(int(n_seg), world_size)
    out, lo = [], 0
    for r in range(world_size):
        hi = lo + base + (1 if r < extra else 0)
        out.append(range(lo, hi))
        lo = hi
    return out


def gather_segments(local: torch.Tensor, owned: List[range], group=None) -> torch.Tensor:
    """All-gather of per-segment tensors: every rank passes its own block [len(owned[rank]), ...]
    and gets [n_seg, ...] in segment order.  Blocks differ in size by at most one, so each is sent
    padded to the largest and trimmed on arrival."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    width = max(len(r) for r in owned)
    padded = torch.zeros((width,) + tuple(local.shape[1:]), dtype=local.dtype, device=local.device)
    padded[: local.shape[0]] = local
    bufs = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(bufs, padded, group=group)
    return torch.cat([bufs[r][: len(owned[r])] for r in range(world)], 0)


class _LibraryBackend:
    """The library's calls on one device and stream: the compute of every pass."""

    def __init__(self, device, stream):
        self.device, self.stream = device, stream

    def prefill(self, q, k, v, g, beta, cu, init):
        out, fin, _ = prefill(q, k, v, g, beta, cu, init, final_state=True, stream=self.stream)
        return out, fin

    def scan(self, s_loc, m, seq_seg, s_start):
        """The scan; returns every sequence's final state."""
        fin = torch.empty((len(seq_seg) - 1,) + tuple(s_loc.shape[1:]), device=s_loc.device,
                          dtype=s_loc.dtype)
        cp_combine(s_loc, m, seq_seg, s_start, final_state=fin, stream=self.stream)
        return fin

    def correct(self, out, u, s_start, cu, skip):
        return cp_correct(out, u, s_start, cu, skip, stream=self.stream)


def _prefill_cp_ranks(q, k, v, g, beta, lengths, init_state, seg_len, backend, group=None):
    """The rank-local part of a context-parallel prefill (see prefill_cp_distributed); `backend`
    supplies the prefill of a varlen batch and the segment scan."""
    import torch.distributed as dist

    rank, world = dist.get_rank(group), dist.get_world_size(group)
    T, H, D = q.shape
    N = len(lengths)
    bounds, seq_seg = segments(lengths, seg_len)
    n_seg = len(bounds)
    owned = assign_segments(n_seg, world)
    mine = owned[rank]
    # states in the initial states' precision (fp32 on the library's path)
    dev, f32 = q.device, (init_state.dtype if init_state is not None else torch.float32)
    # a sequence's first segment starts from the sequence's own initial state
    first_of = {seq_seg[n]: n for n in range(N)}
    tok_lo = bounds[mine.start][0] if len(mine) else 0
    tok_hi = bounds[mine.stop - 1][1] if len(mine) else 0
    if len(mine):
        sl = slice(tok_lo, tok_hi)
        xq, xk, xv, xg, xb = q[sl], k[sl], v[sl], g[sl], beta[sl]
        cu = torch.tensor([bounds[j][0] - tok_lo for j in mine] + [tok_hi - tok_lo], dtype=torch.int32,
                          device=dev)
        init = torch.zeros((len(mine), H, D, D), device=dev, dtype=f32)
        for j in mine:
            if j in first_of and init_state is not None:
                init[j - mine.start] = init_state[first_of[j]]
        # 1. own segments from their local starts: o_loc and S_loc;  2. with v = 0 from the
        # identity: u and M
        o_mine, s_loc_mine = backend.prefill(xq, xk, xv, xg, xb, cu, init)
        eye = torch.eye(D, device=dev, dtype=f32).expand(len(mine), H, D, D).contiguous()
        u_mine, m_mine = backend.prefill(xq, xk, torch.zeros_like(xv), xg, xb, cu, eye)
    else:
        s_loc_mine = torch.zeros((0, H, D, D), device=dev, dtype=f32)
        m_mine = torch.zeros((0, H, D, D), device=dev, dtype=f32)
    # the exchange: every segment's map and local end state on every rank
    s_loc = gather_segments(s_loc_mine, owned, group)
    m = gather_segments(m_mine, owned, group)
    # 3. the scan over all segments: true start states (a first segment keeps its initial state)
    s_start = torch.zeros((n_seg, H, D, D), device=dev, dtype=f32)
    if init_state is not None:
        for j, n in first_of.items():
            s_start[j] = init_state[n]
    fin_all = backend.scan(s_loc, m, seq_seg, s_start)
    # 4. the outputs of the own tokens (a segment that starts its sequence is already exact), and
    # the final state of every sequence whose last segment is here
    out_mine, finals = None, {}
    if len(mine):
        skip = [j - mine.start for j in mine if j in first_of]
        out_mine = backend.correct(o_mine, u_mine, s_start[mine.start:mine.stop].contiguous(), cu, skip)
        for n in range(N):
            if seq_seg[n + 1] - 1 in mine:
                finals[n] = fin_all[n]
    return out_mine, (tok_lo, tok_hi), finals


def prefill_cp_distributed(q, k, v, g, beta, init_state=None, *, seg_len: int, lengths: Sequence[int],
                           group=None, stream=None):
    """Context-parallel prefill across the ranks of a torch.distributed group (one GPU each).

    Every rank passes the same packed inputs (q, k, v, g, beta on its own device; init_state fp32
    [N, H, 128, 128] or None) and the same `lengths` and `seg_len`.  The sequences are cut into
    segments of `seg_len` tokens; rank r prefills the r-th contiguous block of them (passes 1 and
    2), one all-gather shares every segment's (M, S_loc) (the only exchange, 2 x H x 128 x 128 fp32
    per segment), and every rank runs the scan and the output correction over its own block.  Returns
    (out, (t0, t1), finals): the outputs of the rank's tokens t0..t1-1 (fp32 [t1 - t0, H, 128]),
    and {sequence index: final state [H, 128, 128]} for the sequences ending on this rank."""
    dev = q.device
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    lengths = [int(L) for L in lengths]
    if sum(lengths) != q.shape[0]:
        raise ValueError("lengths do not add up to the token count")
    with torch.cuda.stream(s):
        return _prefill_cp_ranks(q, k, v, g, beta, lengths, init_state, seg_len, _LibraryBackend(dev, s), group)
