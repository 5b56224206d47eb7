"""GB300-native Kimi Delta Attention (KDA): thin torch binding over the C ABI of libkda_gb300.

The three calls of the path (and the cross-check path), and the pre-mixer and output gate around
it, mirror include/kda.h.  This module only checks
tensor properties, allocates outputs with torch when the caller does not pass them, and
hands raw device pointers plus the current CUDA stream to the library; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: without the
built library or a CUDA device the calls raise.

Recurrence ("Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA"):
per head S' = diag(exp(clamp(g_t,-5,0))) S_{t-1}, S_t = S' + beta_t k_t (v_t - S'^T k_t)^T,
o_t = S_t^T q_t.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import KDAError

__all__ = ["prefill", "prefill_recurrent", "decode", "state_copy", "device_status", "prefill_path",
           "num_checkpoints", "KDAError", "load", "diag_device_timeout", "premix", "output_gate",
           "prefill_staged"]

_DTYPES = {torch.bfloat16: _lib.KDA_BF16, torch.float32: _lib.KDA_F32}


def load():
    """Load libkda_gb300.so (raises if it is not built)."""
    return _lib.load()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require(t: torch.Tensor, name: str, device, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def num_checkpoints(lengths: Sequence[int], ckpt_stride: int) -> int:
    """Checkpoint slots a prefill emits: sum over sequences of floor(len / stride)."""
    return 0 if ckpt_stride <= 0 else int(sum(int(L) // ckpt_stride for L in lengths))


def prefill_path(d_k: int = 128, d_v: int = 128, dtype=torch.bfloat16) -> int:
    """1 = tensor-core chunked kernel, 0 = per-token CUDA-core kernel, <0 = unsupported."""
    return int(_lib.load().kda_prefill_path(d_k, d_v, _DTYPES[dtype]))


def _prefill(fn_name, q, k, v, g, beta, cu_seqlens, init_state, out, final_state, ckpt_stride,
             ckpts, lengths, stream, out_dtype):
    lib = _lib.load()
    dev = q.device
    dtype = q.dtype
    if dtype not in _DTYPES:
        raise ValueError("q/k/v/g/beta must be bfloat16 or float32")
    T, H, dk = q.shape
    dv = v.shape[-1]
    for t, name, shp in ((q, "q", (T, H, dk)), (k, "k", (T, H, dk)), (g, "g", (T, H, dk)),
                         (v, "v", (T, H, dv)), (beta, "beta", (T, H))):
        _require(t, name, dev, dtype, shp)
    if cu_seqlens is None:
        n = 1
    else:
        _require(cu_seqlens, "cu_seqlens", dev, torch.int32)
        n = cu_seqlens.numel() - 1
    if init_state is not None:
        _require(init_state, "init_state", dev, torch.float32, (n, H, dk, dv))
    if out_dtype not in _DTYPES:
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((T, H, dv), device=dev, dtype=out_dtype)
    else:
        _require(out, "out", dev, out_dtype, (T, H, dv))
    if final_state is True:
        final_state = torch.empty((n, H, dk, dv), device=dev, dtype=torch.float32)
    elif final_state is False or final_state is None:
        final_state = None
    else:
        _require(final_state, "final_state", dev, torch.float32, (n, H, dk, dv))
    if lengths is not None and (len(lengths) != n or sum(int(L) for L in lengths) != T):
        raise ValueError(f"lengths must hold {n} sequence lengths adding up to {T}")
    if ckpt_stride:
        if lengths is None:  # host read of the lengths (synchronizes); pass `lengths` to avoid it
            lengths = [T] if cu_seqlens is None else torch.diff(cu_seqlens).tolist()
        slots = num_checkpoints(lengths, ckpt_stride)
        if ckpts is None:
            ckpts = torch.empty((slots, H, dk, dv), device=dev, dtype=torch.float32)
        else:   # the kernel writes every slot the sequences reach: a smaller buffer would overflow
            _require(ckpts, "ckpts", dev, torch.float32)
            if ckpts.dim() != 4 or tuple(ckpts.shape[1:]) != (H, dk, dv) or ckpts.shape[0] < slots:
                raise ValueError(f"ckpts must be [>= {slots}, {H}, {dk}, {dv}] (got {tuple(ckpts.shape)})")
    elif ckpts is not None:
        _require(ckpts, "ckpts", dev, torch.float32)
    if ckpts is not None and ckpts.numel() == 0:
        ckpt_stride = 0   # no sequence reaches a checkpoint: nothing to emit
    rc = getattr(lib, fn_name)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), n, T, H, dk, dv,
        _DTYPES[dtype], _DTYPES[out_dtype], _ptr(init_state), _ptr(out), _ptr(final_state),
        int(ckpt_stride),
        _ptr(ckpts), _stream(dev, stream))
    _lib.check(rc, fn_name)
    return out, final_state, ckpts


def prefill(q, k, v, g, beta, cu_seqlens=None, init_state=None, *, out=None, final_state=True,
            ckpt_stride: int = 0, ckpts=None, lengths=None, stream=None, out_dtype=torch.float32,
            precise: bool = False):
    """Varlen chunked KDA prefill (kda_prefill, or kda_prefill_precise with precise=True).

    q, k, g: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H] (bf16 or fp32, contiguous, CUDA);
    cu_seqlens: int32 [N+1] on the device or None for one sequence; init_state: fp32
    [N, H, d_k, d_v] or None (zeros).  final_state: True to allocate, a tensor to fill, or
    None/False.  ckpt_stride: 0 or a multiple of 32.  out_dtype: float32 (default, the
    accumulation precision) or bfloat16.  precise: the tensor-core kernel's precise mode (about
    35 % smaller output error, about 1.09x the time).  Returns (out, final_state, ckpts).
    """
    return _prefill("kda_prefill_precise" if precise else "kda_prefill", q, k, v, g, beta,
                    cu_seqlens, init_state, out, final_state, ckpt_stride, ckpts, lengths, stream,
                    out_dtype)


def prefill_recurrent(q, k, v, g, beta, cu_seqlens=None, init_state=None, *, out=None,
                      final_state=True, ckpt_stride: int = 0, ckpts=None, lengths=None, stream=None,
                      out_dtype=torch.float32):
    """Same as prefill, always through the token-by-token CUDA-core kernel."""
    return _prefill("kda_prefill_recurrent", q, k, v, g, beta, cu_seqlens, init_state, out,
                    final_state, ckpt_stride, ckpts, lengths, stream, out_dtype)


def decode(q, k, v, g, beta, state, *, out=None, stream=None, out_dtype=torch.float32):
    """One-token KDA update (kda_decode): state [N, H, d_k, d_v] fp32 is updated in place.
    q, k, g: [N, H, d_k]; v: [N, H, d_v]; beta: [N, H].  Returns out [N, H, d_v] (out_dtype)."""
    lib = _lib.load()
    dev, dtype = q.device, q.dtype
    N, H, dk = q.shape
    dv = v.shape[-1]
    for t, name, shp in ((q, "q", (N, H, dk)), (k, "k", (N, H, dk)), (g, "g", (N, H, dk)),
                         (v, "v", (N, H, dv)), (beta, "beta", (N, H))):
        _require(t, name, dev, dtype, shp)
    _require(state, "state", dev, torch.float32, (N, H, dk, dv))
    if out is None:
        out = torch.empty((N, H, dv), device=dev, dtype=out_dtype)
    else:
        _require(out, "out", dev, out_dtype, (N, H, dv))
    rc = lib.kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                        N, H, dk, dv, _DTYPES[dtype], _DTYPES[out.dtype], _stream(dev, stream))
    _lib.check(rc, "kda_decode")
    return out


def premix(xq, xk, xv, a, b, w, cu_seqlens=None, hist=None, *, eps: float = 1e-6, out=None,
           stream=None):
    """Pre-mixer (kda_premix): the recurrence's inputs from the KDA projections.

    xq, xk, xv, a: [T, H, d]; b: [T, H] (bf16 or fp32, one dtype); w: fp32 [3, H*d, 4], the
    width-4 causal taps of the q, k, v filters (tap 3 on the current token); cu_seqlens: int32
    [N+1] or None; hist: [N, 3, 3, H*d] conv history (the three projected tokens before each
    sequence, per q/k/v) or None for zeros.  Returns (q, k, v, g, beta): q and k L2-normalised
    per (token, head), g = clamp(-softplus(a), -5, 0), beta = sigmoid(b); `out` may pass those
    five tensors preallocated."""
    lib = _lib.load()
    dev, dtype = xq.device, xq.dtype
    if dtype not in _DTYPES:
        raise ValueError("premix inputs must be bfloat16 or float32")
    T, H, d = xq.shape
    for t, name, shp in ((xq, "xq", (T, H, d)), (xk, "xk", (T, H, d)), (xv, "xv", (T, H, d)),
                         (a, "a", (T, H, d)), (b, "b", (T, H))):
        _require(t, name, dev, dtype, shp)
    _require(w, "w", dev, torch.float32, (3, H * d, 4))
    if cu_seqlens is None:
        n = 1
    else:
        _require(cu_seqlens, "cu_seqlens", dev, torch.int32)
        n = cu_seqlens.numel() - 1
    if hist is not None:
        _require(hist, "hist", dev, dtype, (n, 3, 3, H * d))
    if out is None:
        out = tuple(torch.empty_like(xq) for _ in range(4)) + (torch.empty_like(b),)
    else:
        for t, name, shp in zip(out, ("q", "k", "v", "g", "beta"), [(T, H, d)] * 4 + [(T, H)]):
            _require(t, name, dev, dtype, shp)
    rc = lib.kda_premix(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(a), _ptr(b), _ptr(w), _ptr(hist),
                        _ptr(cu_seqlens), n, T, H, d, float(eps), _DTYPES[dtype],
                        *[_ptr(t) for t in out], _stream(dev, stream))
    _lib.check(rc, "kda_premix")
    return tuple(out)


def output_gate(o, z, *, out=None, out_dtype=None, stream=None):
    """Input-dependent output gate (kda_output_gate): out = o * sigmoid(z), elementwise.
    o and z: CUDA tensors of one shape (bf16 or fp32 each).  out: a tensor to fill (may be o
    itself for an in-place gate), else a new one of `out_dtype` (default o.dtype)."""
    lib = _lib.load()
    dev = o.device
    _require(o, "o", dev)
    _require(z, "z", dev, shape=o.shape)
    if o.dtype not in _DTYPES or z.dtype not in _DTYPES:
        raise ValueError("o and z must be bfloat16 or float32")
    if out is None:
        out = torch.empty(o.shape, device=dev, dtype=out_dtype or o.dtype)
    else:
        _require(out, "out", dev, shape=o.shape)
        if out.dtype not in _DTYPES:
            raise ValueError("out must be bfloat16 or float32")
    rc = lib.kda_output_gate(_ptr(o), _DTYPES[o.dtype], _ptr(z), _DTYPES[z.dtype], _ptr(out),
                             _DTYPES[out.dtype], o.numel(), _stream(dev, stream))
    _lib.check(rc, "kda_output_gate")
    return out


def prefill_staged(h_q, h_k, h_v, h_g, h_beta, h_cu_seqlens=None, init_state=None, *,
                   device=None, chunk_tokens: int = 1024, buffers=None, h_out=None,
                   final_state=None, out_dtype=torch.float32, stream=None, static_tables=False):
    """kda_prefill from pinned host memory with the copies overlapped (kda_prefill_staged).

    h_q, h_k, h_v, h_g: pinned CPU [T, H, 128]; h_beta: pinned CPU [T, H] (one dtype, bf16 or
    fp32); h_cu_seqlens: CPU int32 [N+1] (or a list) or None for one sequence; init_state: device
    fp32 [N, H, 128, 128] or None.  `buffers` (device staging, returned, reusable across calls),
    `h_out` (pinned CPU [T, H, 128]) and `final_state` are allocated when not passed.  The work is
    enqueued on `stream`; synchronise it before reading h_out.  static_tables=True takes
    kda_prefill_staged_static (no caller scratch).  Returns (h_out, final_state, buffers)."""
    import numpy as np

    lib = _lib.load()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    dtype = h_q.dtype
    if dtype not in _DTYPES or out_dtype not in _DTYPES:
        raise ValueError("inputs and outputs must be bfloat16 or float32")
    T, H, D = h_q.shape
    if D != 128:
        raise ValueError("the staged prefill takes d_k = d_v = 128")
    for t, name, shp in ((h_q, "h_q", (T, H, D)), (h_k, "h_k", (T, H, D)), (h_v, "h_v", (T, H, D)),
                         (h_g, "h_g", (T, H, D)), (h_beta, "h_beta", (T, H))):
        if t.device.type != "cpu" or (t.numel() and not t.is_pinned()) or not t.is_contiguous() \
                or t.dtype != dtype or tuple(t.shape) != shp:
            raise ValueError(f"{name} must be a pinned, contiguous CPU tensor {shp} of {dtype}")
    cu = None
    if h_cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(h_cu_seqlens.tolist() if hasattr(h_cu_seqlens, "tolist")
                                             else h_cu_seqlens, dtype=np.int32))
    n = 1 if cu is None else cu.shape[0] - 1
    cu_ptr = None if cu is None else cu.ctypes.data
    if init_state is not None:
        _require(init_state, "init_state", dev, torch.float32, (n, H, D, D))
    if final_state is None:
        final_state = torch.empty((n, H, D, D), device=dev, dtype=torch.float32)
    _require(final_state, "final_state", dev, torch.float32, (n, H, D, D))
    if h_out is None:
        h_out = torch.empty((T, H, D), dtype=out_dtype).pin_memory()
    if h_out.device.type != "cpu" or (h_out.numel() and not h_out.is_pinned()) or \
            h_out.dtype != out_dtype or tuple(h_out.shape) != (T, H, D):
        raise ValueError("h_out must be a pinned CPU tensor [T, H, 128] of out_dtype")
    need = int(lib.kda_prefill_staged_scratch(cu_ptr, n, T, int(chunk_tokens)))
    if need < 0:
        raise ValueError("invalid sequences or chunk size")
    if buffers is None:
        buffers = {k: torch.empty_like(t, device=dev) for k, t in
                   (("q", h_q), ("k", h_k), ("v", h_v), ("g", h_g), ("beta", h_beta))}
        buffers["out"] = torch.empty((T, H, D), device=dev, dtype=out_dtype)
    else:   # staging buffers of an earlier call: they must hold this call's tokens
        for key, ref, dt in (("q", h_q, dtype), ("k", h_k, dtype), ("v", h_v, dtype),
                             ("g", h_g, dtype), ("beta", h_beta, dtype), ("out", h_out, out_dtype)):
            buf = buffers.get(key)
            _require(buf, f"buffers[{key!r}]", dev, dt)
            if buf.numel() < ref.numel():
                raise ValueError(f"buffers[{key!r}] holds {buf.numel()} elements, {ref.numel()} needed")
    head = [_ptr(h_q), _ptr(h_k), _ptr(h_v), _ptr(h_g), _ptr(h_beta), cu_ptr, n, T, H, _DTYPES[dtype],
            _DTYPES[out_dtype], _ptr(init_state)] + \
        [_ptr(buffers[k]) for k in ("q", "k", "v", "g", "beta", "out")] + [_ptr(h_out), _ptr(final_state)]
    if static_tables:   # the library's own table array: no scratch from the caller
        rc = lib.kda_prefill_staged_static(*head, int(chunk_tokens), _stream(dev, stream))
        _lib.check(rc, "kda_prefill_staged_static")
        return h_out, final_state, buffers
    if "scratch" not in buffers or buffers["scratch"].numel() < need:
        buffers["scratch"] = torch.empty(max(need, 1), device=dev, dtype=torch.int32)
    rc = lib.kda_prefill_staged(*head, _ptr(buffers["scratch"]), buffers["scratch"].numel(),
                                int(chunk_tokens), _stream(dev, stream))
    _lib.check(rc, "kda_prefill_staged")
    return h_out, final_state, buffers


def state_copy(dst, src, dst_idx=None, src_idx=None, n: Optional[int] = None, stream=None):
    """dst[dst_idx[i]] = src[src_idx[i]] over whole states (kda_state_copy).
    dst, src: fp32 [slots, H, d_k, d_v]; indices: int64 device tensors or None (identity)."""
    lib = _lib.load()
    dev = dst.device
    _require(dst, "dst", dev, torch.float32)
    _require(src, "src", dev, torch.float32)
    if dst.shape[1:] != src.shape[1:] or dst.dim() != 4:
        raise ValueError("dst and src must be [slots, H, d_k, d_v] with the same H, d_k, d_v")
    for t, name in ((dst_idx, "dst_idx"), (src_idx, "src_idx")):
        if t is not None:
            _require(t, name, dev, torch.int64)
    if n is None:
        n = (dst_idx.numel() if dst_idx is not None else
             src_idx.numel() if src_idx is not None else min(dst.shape[0], src.shape[0]))
    # the kernel reads n entries of each index array (whose length the C call does not take)
    for t, name in ((dst_idx, "dst_idx"), (src_idx, "src_idx")):
        if t is not None and int(n) > t.numel():
            raise ValueError(f"n = {n} exceeds the {t.numel()} entries of {name}")
    _, H, dk, dv = dst.shape
    rc = lib.kda_state_copy(_ptr(dst), _ptr(dst_idx), dst.shape[0], _ptr(src), _ptr(src_idx),
                            src.shape[0], int(n), H, dk, dv, _stream(dev, stream))
    _lib.check(rc, "kda_state_copy")
    return dst


def device_status(stream=None, device=None) -> int:
    """Synchronize and read-and-clear the library's sticky device error word (0 = OK)."""
    import ctypes

    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = ctypes.c_int32(0)
    _lib.check(lib.kda_device_status(ctypes.byref(st), _stream(dev, stream)), "kda_device_status")
    return int(st.value)


def diag_device_timeout(timeout_cycles: int = 2_000_000, stream=None, device=None) -> None:
    """Enqueue the library's failure-detection check: one CTA whose bounded device wait expires
    after `timeout_cycles` SM cycles and records KDA_ERR_DEVICE_TIMEOUT, read back (and cleared)
    by device_status()."""
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _lib.check(lib.kda_diag_device_timeout(int(timeout_cycles), _stream(dev, stream)),
               "kda_diag_device_timeout")
