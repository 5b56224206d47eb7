"""Pins for the fp64 oracle: facts fixed by the recurrence's definition and by mathematics,
not by the oracle itself.

Every pin takes an oracle handle and raises AssertionError when the handle disagrees with
the fact.  ``test_oracle_pins.py`` runs them on the committed oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with a planted mistake and requires each copy to fail one.

Recurrence pinned (page "Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und
globale MLA"): per head S_t = S' + beta_t k_t (v_t - S'^T k_t)^T with S' = diag(exp(g_t)) S_{t-1},
g clamped to [-5, 0]; the read o_t = S_t^T q_t follows the token's own write.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def random_case(seed, T, H=2, dk=8, dv=6, lengths=None, init=True, decay=1.0):
    """Small random fp64 inputs with the workloads' distributions (dimensions kept tiny)."""
    r = _rng(seed)
    lengths = lengths or [T]
    T = sum(lengths)
    q = _unit_rows(r.standard_normal((T, H, dk)))
    k = _unit_rows(r.standard_normal((T, H, dk)))
    v = r.standard_normal((T, H, dv))
    g = np.clip(-np.log1p(np.exp(r.standard_normal((T, H, dk)))), -5, 0) * decay
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    N = len(lengths)
    S0 = 0.05 * r.standard_normal((N, H, dk, dv)) if init else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=S0, cu_seqlens=cu)


def _rel(a, b):
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rhs = line.split("=", 1)
            vals[key.strip()] = np.array([float(x) for x in rhs.split()])
    return vals


# ---------------------------------------------------------------------------------------------


def pin_golden_scalar(orc):
    """Hand-worked 5-token scalar case (tests/golden/scalar_d1.txt): decay, clamp at both
    ends, delta write, read after write."""
    gv = _read_golden("scalar_d1.txt")
    T = len(gv["k"])
    sh = (T, 1, 1)
    out, fin, _ = orc.prefill(gv["q"].reshape(sh), gv["k"].reshape(sh), gv["v"].reshape(sh),
                              gv["g"].reshape(sh), gv["beta"].reshape(T, 1))
    assert np.allclose(out.reshape(-1), gv["out"], rtol=1e-14, atol=1e-16), (out.reshape(-1), gv["out"])
    assert np.allclose(fin.reshape(-1), gv["final"], rtol=1e-14, atol=1e-16)


def pin_golden_two_channel(orc):
    """Hand-worked 2x2 case (tests/golden/hand_d2.txt): key-axis decay, S^T read."""
    gv = _read_golden("hand_d2.txt")
    T = 2
    out, fin, _ = orc.prefill(gv["q"].reshape(T, 1, 2), gv["k"].reshape(T, 1, 2),
                              gv["v"].reshape(T, 1, 2), gv["g"].reshape(T, 1, 2),
                              gv["beta"].reshape(T, 1), init_state=gv["S0"].reshape(1, 1, 2, 2))
    assert np.allclose(out.reshape(-1), gv["out"], rtol=1e-14, atol=1e-15), out.reshape(-1)
    assert np.allclose(fin.reshape(-1), gv["final"], rtol=1e-14, atol=1e-15), fin.reshape(-1)


def pin_identity_gates(orc):
    """beta = 0 and g = 0: the state never changes (bit for bit) and o_t = S_0^T q_t."""
    c = random_case(1, 37, H=3)
    c["beta"][:] = 0.0
    c["g"][:] = 0.0
    out, fin, _ = orc.prefill(**c)
    assert np.array_equal(fin, c["init_state"])
    expect = np.einsum("hij,thi->thj", c["init_state"][0], c["q"])
    assert _rel(out, expect) < 1e-13


def pin_single_token_from_zero(orc):
    """One token from the zero state: S_1 = beta k v^T and o_1 = beta (k.q) v, for any g."""
    c = random_case(2, 1, H=4, init=False)
    out, fin, _ = orc.prefill(**c)
    b = c["beta"][0]
    S1 = b[:, None, None] * np.einsum("hi,hj->hij", c["k"][0], c["v"][0])
    assert _rel(fin[0], S1) < 1e-14
    o1 = (b * np.einsum("hi,hi->h", c["k"][0], c["q"][0]))[:, None] * c["v"][0]
    assert _rel(out[0], o1) < 1e-13


def pin_exact_retrieval(orc):
    """beta = 1 and |k_t| = 1: right after token t, S_t^T k_t = v_t (every state is emitted as a
    checkpoint with stride 1)."""
    c = random_case(3, 25, H=2, dk=8, dv=5)
    c["beta"][:] = 1.0
    _, _, ck = orc.prefill(**c, ckpt_stride=1)
    got = np.einsum("thij,thi->thj", ck, c["k"])
    assert _rel(got, c["v"]) < 1e-12


def pin_orthonormal_keys(orc):
    """g = 0, beta = 1, zero start, keys t = 0..dk-1 from one random orthonormal basis: every
    write lands in an empty direction, so S_T = sum_t k_t v_t^T, and reading with q = k_s
    returns v_s once token s has been written and 0 before."""
    r = _rng(4)
    dk, dv = 6, 4
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Qm.T.copy()                       # rows are orthonormal
    T = dk
    q = np.empty((T, 1, dk))
    q[:, 0] = keys[(np.arange(T) + 2) % dk]  # query a key written two tokens later / earlier
    k = keys.reshape(T, 1, dk)
    v = r.standard_normal((T, 1, dv))
    out, fin, _ = orc.prefill(q, k, v, np.zeros((T, 1, dk)), np.ones((T, 1)))
    assert _rel(fin[0, 0], np.einsum("ti,tj->ij", keys, v[:, 0])) < 1e-13
    for t in range(T):
        s = (t + 2) % dk
        expect = v[s, 0] if s <= t else np.zeros(dv)
        assert np.allclose(out[t, 0], expect, atol=1e-13), (t, out[t, 0], expect)


def pin_decay_only(orc):
    """beta = 0 with random g: S_t = diag(exp(sum_{u<=t} clamp(g_u))) S_0 on the key axis, and
    o_t = S_t^T q_t.  g is drawn beyond both ends of [-5, 0] so the clamp matters."""
    c = random_case(5, 19, H=2, dk=7, dv=5)
    c["beta"][:] = 0.0
    c["g"] = _rng(6).uniform(-7.0, 1.0, size=c["g"].shape)
    out, fin, _ = orc.prefill(**c)
    G = np.cumsum(np.clip(c["g"], -5.0, 0.0), axis=0)       # [T, H, dk]
    St = np.exp(G)[:, :, :, None] * c["init_state"][0][None]
    assert _rel(fin[0], St[-1]) < 1e-13
    assert _rel(out, np.einsum("thij,thi->thj", St, c["q"])) < 1e-13


def pin_transition_form(orc):
    """The recurrence rewritten as an affine map of the state,
    S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T, evaluated with dense
    matrices on a tiny case (a rearrangement, not the oracle's loop)."""
    c = random_case(7, 9, H=1, dk=4, dv=3)
    out, fin, _ = orc.prefill(**c)
    S = c["init_state"][0, 0].copy()
    dk = S.shape[0]
    for t in range(9):
        kk, vv, qq, b = c["k"][t, 0], c["v"][t, 0], c["q"][t, 0], c["beta"][t, 0]
        alpha = np.exp(np.clip(c["g"][t, 0], -5.0, 0.0))
        M = (np.eye(dk) - b * np.outer(kk, kk)) @ np.diag(alpha)
        S = M @ S + b * np.outer(kk, vv)
        assert _rel(out[t, 0], S.T @ qq) < 1e-12
    assert _rel(fin[0, 0], S) < 1e-12


def pin_linearity(orc):
    """For fixed q, k, g, beta the outputs and states are jointly linear in (V, S_0)."""
    c1 = random_case(8, 21, H=2)
    c2 = random_case(9, 21, H=2)
    for key in ("q", "k", "g", "beta"):
        c2[key] = c1[key]
    a, b = 0.7, -1.3
    c3 = dict(c1)
    c3["v"] = a * c1["v"] + b * c2["v"]
    c3["init_state"] = a * c1["init_state"] + b * c2["init_state"]
    o1, f1, _ = orc.prefill(**c1)
    o2, f2, _ = orc.prefill(**c2)
    o3, f3, _ = orc.prefill(**c3)
    assert _rel(o3, a * o1 + b * o2) < 1e-12
    assert _rel(f3, a * f1 + b * f2) < 1e-12


def pin_value_permutation(orc):
    """Permuting the value channels of v and S_0 permutes the columns of o and S the same way."""
    c = random_case(10, 17, H=2, dk=5, dv=7)
    perm = _rng(11).permutation(7)
    o1, f1, _ = orc.prefill(**c)
    c2 = dict(c)
    c2["v"] = c["v"][:, :, perm]
    c2["init_state"] = c["init_state"][:, :, :, perm]
    o2, f2, _ = orc.prefill(**c2)
    assert np.array_equal(o2, o1[:, :, perm])
    assert np.array_equal(f2, f1[:, :, :, perm])


def pin_chunked_agrees(orc):
    """Token-by-token and chunked evaluation agree to 1e-12 (relative) on tiny inputs, for
    several chunk lengths, ragged varlen batches and a nonzero start state."""
    for T in (1, 15, 16, 17, 48, 64):
        c = random_case(100 + T, T, H=2)
        ref, fref, _ = orc.prefill(**c)
        for C in (1, 4, 16, 64):
            out, fin, _ = orc.prefill(**c, chunk=C)
            assert _rel(out, ref) < 1e-12, (T, C, _rel(out, ref))
            assert _rel(fin, fref) < 1e-12, (T, C)
    c = random_case(99, 0, H=3, lengths=[5, 33, 1, 16, 0, 40])
    ref, fref, ck = orc.prefill(**c, ckpt_stride=16)
    out, fin, ck2 = orc.prefill(**c, chunk=16, ckpt_stride=16)
    assert _rel(out, ref) < 1e-12 and _rel(fin, fref) < 1e-12 and _rel(ck2, ck) < 1e-12


def pin_prefix_split(orc):
    """Resuming from the state after a prefix gives the uninterrupted result, and checkpoint m
    equals the final state of the prefix of m*stride tokens."""
    c = random_case(12, 40, H=2)
    out, fin, ck = orc.prefill(**c, ckpt_stride=8)
    assert ck.shape[0] == 5
    for a in (1, 8, 23, 39):
        pre = {key: c[key][:a] for key in ("q", "k", "v", "g", "beta")}
        o_a, s_a, _ = orc.prefill(**pre, init_state=c["init_state"])
        post = {key: c[key][a:] for key in ("q", "k", "v", "g", "beta")}
        o_b, s_b, _ = orc.prefill(**post, init_state=s_a)
        assert _rel(np.concatenate([o_a, o_b]), out) < 1e-13
        assert _rel(s_b, fin) < 1e-13
    for m in range(1, 6):
        pre = {key: c[key][: 8 * m] for key in ("q", "k", "v", "g", "beta")}
        _, s_m, _ = orc.prefill(**pre, init_state=c["init_state"])
        assert np.array_equal(ck[m - 1], s_m[0])


def pin_varlen_packing(orc):
    """A packed varlen batch equals one call per sequence (including empty sequences), and
    checkpoint slots are laid out sequence by sequence."""
    lengths = [7, 0, 20, 3, 16]
    c = random_case(13, 0, H=2, lengths=lengths)
    out, fin, ck = orc.prefill(**c, ckpt_stride=4)
    cu = c["cu_seqlens"]
    slot = 0
    for n, L in enumerate(lengths):
        sl = slice(cu[n], cu[n + 1])
        one = {key: c[key][sl] for key in ("q", "k", "v", "g", "beta")}
        o, f, ckn = orc.prefill(**one, init_state=c["init_state"][n:n + 1], ckpt_stride=4)
        assert np.array_equal(o, out[sl])
        assert np.array_equal(f[0], fin[n])
        nck = L // 4
        if nck:
            assert np.array_equal(ckn, ck[slot:slot + nck])
        slot += nck
    assert ck.shape[0] == slot


def pin_decode_is_one_step(orc):
    """Decode of token t from the state after token t-1 equals row t of a prefill."""
    c = random_case(14, 12, H=3)
    out, fin, ck = orc.prefill(**c, ckpt_stride=1)
    for t in (1, 5, 11):
        o, S = orc.decode(c["q"][t:t + 1], c["k"][t:t + 1], c["v"][t:t + 1], c["g"][t:t + 1],
                          c["beta"][t:t + 1], ck[t - 1:t])
        assert np.array_equal(o[0], out[t])
        assert np.array_equal(S[0], ck[t])


def pin_tile_decay_floor(orc):
    """With g at the floor everywhere a 16-token tile's cumulative log-decay is exactly -80,
    and values below the floor behave as the floor (the clamp)."""
    c = random_case(15, 32, H=1, dk=4, dv=3)
    c["beta"][:] = 0.0
    c["g"][:] = -5.0
    _, f1, _ = orc.prefill(**c)
    c["g"][:] = -9.0
    _, f2, _ = orc.prefill(**c)
    assert np.array_equal(f1, f2)
    assert _rel(f1[0], math.exp(-160.0) * c["init_state"][0]) < 1e-12


# ---- pre-mixer and output gate ------------------------------------------------------------------
# Page "Kimi K3 im Detail", section "Sequenz-Mixing: KDA-Zustand und globale MLA": a short
# convolution of width 4 on the KDA projections (first paragraph) and an input-dependent output
# gate on the mixer's output (third paragraph).  The readings the oracle takes (causal depthwise
# taps, zero or given history, q/k L2 normalisation, g = clamp(-softplus(a), -5, 0),
# beta = sigmoid(b), out = o * sigmoid(z)) are pinned here by a hand-worked case, closed forms and
# invariants.


def premix_case(seed, lengths, H=2, d=8, hist=False):
    r = _rng(seed)
    T = sum(lengths)
    x = [r.standard_normal((T, H, d)) for _ in range(3)]
    a = r.standard_normal((T, H, d))
    b = r.standard_normal((T, H))
    w = r.standard_normal((3, H * d, 4))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    hs = r.standard_normal((len(lengths), 3, 3, H * d)) if hist else None
    return dict(xq=x[0], xk=x[1], xv=x[2], a=a, b=b, w=w, hist=hs, cu_seqlens=cu)


def pin_premix_golden(orc):
    gv = _read_golden("premix_d2.txt")
    x = gv["x"].reshape(6, 1, 2)
    w = np.stack([gv[n].reshape(2, 4) for n in ("wq", "wk", "wv")])
    q, k, v, g, beta = orc.premix(x, x, x, gv["a"].reshape(6, 1, 2), gv["b"].reshape(6, 1), w,
                                  cu_seqlens=gv["cu"].astype(np.int64))
    for name, got in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        assert np.allclose(got.ravel(), gv[name], rtol=0, atol=1e-12), name


def pin_premix_current_tap_only(orc):
    # taps (0, 0, 0, 1): v is the projection itself, q and k its per-head unit vectors
    c = premix_case(41, [7, 3], H=3)
    c["w"][:] = [0.0, 0.0, 0.0, 1.0]
    q, k, v, _, _ = orc.premix(**c)
    assert np.array_equal(v, c["xv"])
    assert _rel(q, _unit_rows(c["xq"])) < 1e-14 and _rel(k, _unit_rows(c["xk"])) < 1e-14


def pin_premix_shift_resets_per_sequence(orc):
    # taps (0, 0, 1, 0): v_t = x_(t-1) inside a sequence, zero on every sequence's first token
    lengths = [5, 1, 7]
    c = premix_case(42, lengths)
    c["w"][:] = [0.0, 0.0, 1.0, 0.0]
    _, _, v, _, _ = orc.premix(**c)
    cu = c["cu_seqlens"]
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        assert np.all(v[s] == 0.0)
        assert np.array_equal(v[s + 1:e], c["xv"][s:e - 1])


def pin_premix_history_is_a_prefix(orc):
    # history rows h = the three tokens before the sequence: same as prefilling them and dropping
    # their outputs (also for sequences shorter than the window)
    for L in (1, 2, 6):
        c = premix_case(43 + L, [L], hist=True)
        H, d = c["xq"].shape[1:]
        longer = {}
        for i, name in enumerate(("xq", "xk", "xv")):
            pre = c["hist"][0, i].reshape(3, H, d)
            longer[name] = np.concatenate([pre, c[name]])
        a = np.concatenate([np.zeros((3, H, d)), c["a"]])
        b = np.concatenate([np.zeros((3, H)), c["b"]])
        ref = orc.premix(longer["xq"], longer["xk"], longer["xv"], a, b, c["w"])
        got = orc.premix(**c)
        for x, y in zip(got, ref):
            assert _rel(x, y[3:]) < 1e-14


def pin_premix_varlen_packing(orc):
    lengths = [4, 9, 2]
    c = premix_case(47, lengths, hist=True)
    packed = orc.premix(**c)
    cu = c["cu_seqlens"]
    for n in range(len(lengths)):
        s, e = cu[n], cu[n + 1]
        one = orc.premix(c["xq"][s:e], c["xk"][s:e], c["xv"][s:e], c["a"][s:e], c["b"][s:e],
                         c["w"], hist=c["hist"][n:n + 1])
        for x, y in zip(packed, one):
            assert np.array_equal(x[s:e], y)


def pin_premix_conv_is_linear_and_scale_free(orc):
    c = premix_case(48, [11])
    q1, k1, v1, _, _ = orc.premix(**c)
    c2 = dict(c, xq=3.5 * c["xq"], xk=0.25 * c["xk"], xv=c["xv"] + c["xq"])
    q2, k2, v2, _, _ = orc.premix(**c2)
    c3 = dict(c, xv=c["xq"])
    _, _, v3, _, _ = orc.premix(**c3)
    assert _rel(q2, q1) < 1e-14 and _rel(k2, k1) < 1e-14            # positive scaling is undone
    assert _rel(v2, v1 + v3) < 1e-14                                 # the convolution is linear
    assert np.allclose(np.linalg.norm(q1, axis=-1), 1.0, atol=1e-14)


def pin_premix_gates(orc):
    cs = np.array([0.01, 0.5, 1.0, 2.5, 4.0, 4.999])
    c = premix_case(49, [len(cs)], H=1, d=1)
    c["a"] = np.log(np.expm1(cs)).reshape(-1, 1, 1)               # softplus(a) = c exactly
    c["b"] = np.array([-3.0, -1.0, 0.0, 0.5, 1.0, 3.0]).reshape(-1, 1)
    _, _, _, g, beta = orc.premix(**c)
    assert np.allclose(g.ravel(), -cs, rtol=0, atol=1e-13)
    c_neg = dict(c, b=-c["b"])
    _, _, _, _, beta_neg = orc.premix(**c_neg)
    assert np.allclose(beta + beta_neg, 1.0, rtol=0, atol=1e-15)    # sigmoid(-b) = 1 - sigmoid(b)
    c_big = dict(c, a=np.full_like(c["a"], 5.5))                     # softplus(5.5) > 5: clamped
    _, _, _, g_big, _ = orc.premix(**c_big)
    assert np.all(g_big == -5.0)


def pin_output_gate(orc):
    r = _rng(50)
    o = r.standard_normal((6, 2, 8))
    assert np.array_equal(orc.output_gate(o, np.zeros_like(o)), o / 2)
    l3 = np.full_like(o, math.log(3.0))
    assert np.allclose(orc.output_gate(o, l3), 0.75 * o, rtol=1e-15, atol=0)
    assert np.allclose(orc.output_gate(o, -l3), 0.25 * o, rtol=1e-15, atol=0)
    z = r.standard_normal(o.shape)
    assert np.allclose(orc.output_gate(o, z) + orc.output_gate(o, -z), o, rtol=0, atol=1e-15)
    assert np.allclose(orc.output_gate(o, np.full_like(o, 50.0)), o, rtol=1e-15, atol=0)


PINS = [
    pin_golden_scalar,
    pin_golden_two_channel,
    pin_identity_gates,
    pin_single_token_from_zero,
    pin_exact_retrieval,
    pin_orthonormal_keys,
    pin_decay_only,
    pin_transition_form,
    pin_linearity,
    pin_value_permutation,
    pin_chunked_agrees,
    pin_prefix_split,
    pin_varlen_packing,
    pin_decode_is_one_step,
    pin_tile_decay_floor,
    pin_premix_golden,
    pin_premix_current_tap_only,
    pin_premix_shift_resets_per_sequence,
    pin_premix_history_is_a_prefix,
    pin_premix_varlen_packing,
    pin_premix_conv_is_linear_and_scale_free,
    pin_premix_gates,
    pin_output_gate,
]
