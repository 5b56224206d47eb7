"""fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product (the CUDA library and its binding) never does; the two
share no code.  The arithmetic lives in ``kda_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays.

Source of the computation: "Kimi K3 im Detail" (flozi.net), section "Sequenz-Mixing:
KDA-Zustand und globale MLA" -- per-head recurrent state, channel-wise retention, scalar
delta-rule write gate, read S_t^T q_t after the token's own update, log-decay floor -5; around
it, the width-4 short convolution of the projections and the input-dependent output gate (the
readings taken where the page gives no formula are stated in ``kda_oracle.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "kda_oracle.c")
_DEFAULT_LIB = os.path.join(_HERE, "_build", "libkda_oracle.so")


def build(source: str = SOURCE, out: str = _DEFAULT_LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math: IEEE fp64 throughout). Returns the .so path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    """Exact conversion of a numpy array or a torch tensor (any float dtype) to contiguous fp64."""
    if hasattr(a, "detach"):  # torch tensor: bf16/fp32 -> fp64 is exact
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Oracle:
    """Handle on one compiled copy of the oracle (the tests also load deliberately broken copies)."""

    def __init__(self, libpath: Optional[str] = None):
        self.libpath = libpath or build()
        lib = ctypes.CDLL(self.libpath)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        common = [dp, dp, dp, dp, dp, ip, i64, i64, i64, i64, dp, dp, dp, i64, dp]
        lib.kda_oracle_prefill.argtypes = common + [ctypes.c_int]
        lib.kda_oracle_prefill.restype = ctypes.c_int
        lib.kda_oracle_chunked.argtypes = common + [i64, ctypes.c_int]
        lib.kda_oracle_chunked.restype = ctypes.c_int
        lib.kda_oracle_decode.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64]
        lib.kda_oracle_decode.restype = ctypes.c_int
        lib.kda_oracle_num_ckpts.argtypes = [ip, i64, i64]
        lib.kda_oracle_num_ckpts.restype = i64
        lib.kda_oracle_premix.argtypes = [dp, dp, dp, dp, dp, dp, dp, ip, i64, i64, i64,
                                          ctypes.c_double, dp, dp, dp, dp, dp]
        lib.kda_oracle_premix.restype = ctypes.c_int
        lib.kda_oracle_output_gate.argtypes = [dp, dp, i64, dp]
        lib.kda_oracle_output_gate.restype = ctypes.c_int
        self._lib = lib

    def prefill(self, q, k, v, g, beta, cu_seqlens=None, init_state=None, ckpt_stride: int = 0,
                chunk: int = 0, threads: Optional[int] = None):
        """Run the oracle on packed varlen inputs.

        q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; cu_seqlens: [N+1] (default [0, T]);
        init_state: [N, H, dk, dv] or None (zeros).  chunk=0 evaluates token by token; chunk>0
        uses the independent chunked evaluation.  Returns (out [T,H,dv], final [N,H,dk,dv],
        ckpts [n_ckpt,H,dk,dv] or None), all fp64.
        """
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        T, H, dk = q.shape
        dv = v.shape[2]
        assert k.shape == (T, H, dk) and g.shape == (T, H, dk)
        assert v.shape == (T, H, dv) and beta.shape == (T, H)
        if cu_seqlens is None:
            cu_seqlens = [0, T]
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
        assert cu[0] == 0 and cu[-1] == T
        init = None
        if init_state is not None:
            init = _f64(init_state)
            assert init.shape == (N, H, dk, dv)
        out = np.zeros((T, H, dv))
        final = np.zeros((N, H, dk, dv))
        n_ck = int(self._lib.kda_oracle_num_ckpts(
            cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, int(ckpt_stride)))
        ckpts = np.zeros((n_ck, H, dk, dv)) if n_ck > 0 else None
        nthreads = int(threads or os.cpu_count() or 1)
        args = [_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, H, dk, dv, _ptr(init),
                _ptr(out), _ptr(final), int(ckpt_stride), _ptr(ckpts)]
        if chunk:
            rc = self._lib.kda_oracle_chunked(*args, int(chunk), nthreads)
        else:
            rc = self._lib.kda_oracle_prefill(*args, nthreads)
        if rc != 0:
            raise ValueError(f"oracle prefill failed with code {rc}")
        return out, final, ckpts

    def decode(self, q, k, v, g, beta, state):
        """One-token update of every (sequence, head).  q,k,g [N,H,dk], v [N,H,dv], beta [N,H],
        state [N,H,dk,dv] (not modified).  Returns (out [N,H,dv], new_state), fp64."""
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        S = _f64(state).copy()
        N, H, dk = q.shape
        dv = v.shape[2]
        assert S.shape == (N, H, dk, dv) and beta.shape == (N, H)
        out = np.zeros((N, H, dv))
        rc = self._lib.kda_oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S),
                                         _ptr(out), N, H, dk, dv)
        if rc != 0:
            raise ValueError(f"oracle decode failed with code {rc}")
        return out, S

    def premix(self, xq, xk, xv, a, b, w, hist=None, cu_seqlens=None, eps: float = 1e-6):
        """Short convolution of the q, k, v projections, q/k normalisation and the gates.

        xq, xk, xv, a: [T, H, d]; b: [T, H]; w: [3, H*d, 4] (taps on x_{t-3} .. x_t);
        hist: [N, 3, 3, H*d] or None (zeros); cu_seqlens: [N+1] (default [0, T]).
        Returns (q, k, v, g, beta) in fp64 with the shapes of (xq, xk, xv, a, b)."""
        xq, xk, xv, a, b, w = (_f64(x) for x in (xq, xk, xv, a, b, w))
        T, H, d = xq.shape
        assert xk.shape == xq.shape and xv.shape == xq.shape and a.shape == xq.shape
        assert b.shape == (T, H) and w.shape == (3, H * d, 4)
        if cu_seqlens is None:
            cu_seqlens = [0, T]
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens, dtype=np.int64))
        N = cu.shape[0] - 1
        assert cu[0] == 0 and cu[-1] == T
        hs = None
        if hist is not None:
            hs = _f64(hist)
            assert hs.shape == (N, 3, 3, H * d)
        outs = [np.zeros((T, H, d)) for _ in range(4)] + [np.zeros((T, H))]
        rc = self._lib.kda_oracle_premix(_ptr(xq), _ptr(xk), _ptr(xv), _ptr(a), _ptr(b), _ptr(w),
                                         _ptr(hs), cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                         N, H, d, float(eps), *[_ptr(o) for o in outs])
        if rc != 0:
            raise ValueError(f"oracle premix failed with code {rc}")
        return tuple(outs)

    def output_gate(self, o, z):
        """out = o * sigmoid(z), elementwise, fp64 (o and z of the same shape)."""
        o, z = _f64(o), _f64(z)
        assert o.shape == z.shape
        out = np.zeros(o.shape)
        rc = self._lib.kda_oracle_output_gate(_ptr(o), _ptr(z), o.size, _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle output gate failed with code {rc}")
        return out


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    """The oracle built from the committed source (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def build_variant(source_text: str, workdir: Optional[str] = None) -> Oracle:
    """Compile a modified copy of the oracle source (used by the tests that plant mistakes)."""
    workdir = workdir or tempfile.mkdtemp(prefix="kda_oracle_variant_")
    src = os.path.join(workdir, "kda_oracle.c")
    with open(src, "w") as f:
        f.write(source_text)
    return Oracle(build(src, os.path.join(workdir, "libkda_oracle.so"), force=True))
