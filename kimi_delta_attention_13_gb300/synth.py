"""Seeded synthetic inputs for the KDA prefill / decode workloads.

This module only draws random numbers with torch and shapes them into the input
distributions of the workloads; it holds none of the recurrence's arithmetic.  Both the
CUDA path (through the tests and the benchmark) and the fp64 oracle are fed from here.

Distributions (per workload): q, k ~ N(0,1) then L2-normalised over the head dimension;
v ~ N(0,1); g = clamp(-softplus(N(0,1)), -5, 0) per key channel; beta = sigmoid(N(0,1));
initial states, where used, 0.05 * N(0,1) in fp32.  Draw order from one generator:
q, k, v, g, beta, state.  The head geometry (96 heads of width 128) is the one the
"Kimi K3 im Detail" page gives for KDA (section "Sequenz-Mixing").
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch
import torch.nn.functional as F

HEADS = 96
HEAD_DIM = 128


@dataclass
class Workload:
    """One named workload: shapes, dtype, seed and options."""

    name: str
    kind: str                      # "prefill" or "decode"
    lengths: List[int]             # prefill: per-sequence token counts; decode: [1] * N
    heads: int = HEADS
    d_k: int = HEAD_DIM
    d_v: int = HEAD_DIM
    dtype: str = "bf16"            # input/output dtype: "bf16" or "f32"
    seed: int = 0
    init_state: bool = False
    ckpt_stride: int = 0
    oracle_heads: Optional[List[int]] = None   # heads the oracle checks (None = all)
    notes: str = field(default="")

    @property
    def n_seqs(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))


def varlen8_lengths() -> List[int]:
    """Eight sequence lengths uniform in [1024, 32768], drawn from a CPU generator seeded 2."""
    gen = torch.Generator().manual_seed(2)
    return [int(x) for x in torch.randint(1024, 32769, (8,), generator=gen)]


def long_context_oracle_heads() -> List[int]:
    """The 8 heads (of 96) the oracle checks on the 262,144-token workload (seed 4)."""
    gen = torch.Generator().manual_seed(4)
    return sorted(int(x) for x in torch.randperm(HEADS, generator=gen)[:8])


def workloads() -> List[Workload]:
    """The five workloads, in order: tiny fp32, T=8192, varlen x8, decode x256, T=262144."""
    return [
        Workload("tiny-f32-T64-H2", "prefill", [64], heads=2, dtype="f32", seed=0),
        Workload("prefill-bf16-T8192-H96", "prefill", [8192], seed=1),
        Workload("varlen8-bf16-H96-init", "prefill", varlen8_lengths(), seed=2, init_state=True),
        Workload("decode-bf16-N256-H96", "decode", [1] * 256, seed=3, init_state=True),
        Workload("long-bf16-T262144-H96-ckpt4096", "prefill", [262144], seed=4, ckpt_stride=4096,
                 oracle_heads=long_context_oracle_heads()),
    ]


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_inputs(lengths: List[int], heads: int = HEADS, d_k: int = HEAD_DIM, d_v: int = HEAD_DIM,
                dtype: str = "bf16", seed: int = 0, device="cpu", init_state: bool = False,
                decay_scale: float = 1.0) -> dict:
    """Draw one batch of packed varlen inputs on `device`.

    Returns a dict with q, k, g [T,H,d_k], v [T,H,d_v], beta [T,H] in `dtype`, `state`
    [N,H,d_k,d_v] fp32 (or None) and `cu_seqlens` [N+1] int32 on `device`.
    `decay_scale` multiplies g (0.01 gives slow decay, so the state carries far).
    """
    gen = torch.Generator(device=device).manual_seed(seed)
    T = int(sum(lengths))
    N = len(lengths)
    dt = torch_dtype(dtype)
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    q = _unit(torch.randn(T, heads, d_k, **kw)).to(dt)
    k = _unit(torch.randn(T, heads, d_k, **kw)).to(dt)
    v = torch.randn(T, heads, d_v, **kw).to(dt)
    g = (-F.softplus(torch.randn(T, heads, d_k, **kw))).clamp(-5.0, 0.0)
    if decay_scale != 1.0:
        g = g * decay_scale
    g = g.to(dt)
    beta = torch.sigmoid(torch.randn(T, heads, **kw)).to(dt)
    state = (0.05 * torch.randn(N, heads, d_k, d_v, **kw)) if init_state else None
    cu = torch.zeros(N + 1, dtype=torch.int64)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state=state,
                cu_seqlens=cu.to(device=device, dtype=torch.int32), lengths=list(lengths))


def make_decode_inputs(n_seqs: int, heads: int = HEADS, d_k: int = HEAD_DIM, d_v: int = HEAD_DIM,
                       dtype: str = "bf16", seed: int = 3, device="cpu") -> dict:
    """One new token per sequence plus an fp32 state 0.05*N(0,1): q,k,g [N,H,d_k], v [N,H,d_v],
    beta [N,H], state [N,H,d_k,d_v]."""
    d = make_inputs([1] * n_seqs, heads, d_k, d_v, dtype, seed, device, init_state=True)
    return dict(q=d["q"], k=d["k"], v=d["v"], g=d["g"], beta=d["beta"], state=d["state"])


def make_workload_inputs(w: Workload, device="cpu", decay_scale: float = 1.0) -> dict:
    if w.kind == "decode":
        return make_decode_inputs(w.n_seqs, w.heads, w.d_k, w.d_v, w.dtype, w.seed, device)
    return make_inputs(w.lengths, w.heads, w.d_k, w.d_v, w.dtype, w.seed, device, w.init_state,
                       decay_scale)


def make_premix_inputs(lengths: List[int], heads: int = HEADS, d: int = HEAD_DIM,
                       dtype: str = "bf16", seed: int = 0, device="cpu", hist: bool = False) -> dict:
    """Inputs of the pre-mixer: projection rows xq, xk, xv and the decay pre-activation a, all
    N(0,1) [T,H,d]; the write-gate pre-activation b ~ N(0,1) [T,H]; taps w ~ 0.5 N(0,1) fp32
    [3, H*d, 4]; conv history ~ N(0,1) [N,3,3,H*d] (or None); cu_seqlens int32 [N+1].
    Draw order from one generator: xq, xk, xv, a, b, w, hist.  (The model's projections and
    filter weights are trained; these stand-ins only give the kernels the same shapes.)"""
    gen = torch.Generator(device=device).manual_seed(seed)
    T, N = int(sum(lengths)), len(lengths)
    dt = torch_dtype(dtype)
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    xq, xk, xv, a = (torch.randn(T, heads, d, **kw).to(dt) for _ in range(4))
    b = torch.randn(T, heads, **kw).to(dt)
    w = 0.5 * torch.randn(3, heads * d, 4, **kw)
    hs = torch.randn(N, 3, 3, heads * d, **kw).to(dt) if hist else None
    cu = torch.zeros(N + 1, dtype=torch.int64)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    return dict(xq=xq, xk=xk, xv=xv, a=a, b=b, w=w, hist=hs,
                cu_seqlens=cu.to(device=device, dtype=torch.int32), lengths=list(lengths))


def make_gate_inputs(shape, o_dtype: str = "f32", z_dtype: str = "bf16", seed: int = 0,
                     device="cpu") -> dict:
    """Output-gate inputs: o ~ N(0,1) (the mixer's output) and its gate pre-activation
    z ~ N(0,1), both of `shape`.  Draw order: o, z."""
    gen = torch.Generator(device=device).manual_seed(seed)
    kw = dict(generator=gen, device=device, dtype=torch.float32)
    o = torch.randn(*shape, **kw).to(torch_dtype(o_dtype))
    z = torch.randn(*shape, **kw).to(torch_dtype(z_dtype))
    return dict(o=o, z=z)
