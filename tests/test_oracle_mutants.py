"""Each planted mistake in a copy of the oracle must make at least one pin fail.

The mistakes are the plausible ones: a flipped sign, a dropped term or gate, a decay on the
wrong axis, a read before the write, a transposed read, a wrong operand, a missing clamp,
a causal mask without its diagonal; around the recurrence, reversed convolution taps, a
convolution history that leaks across sequences, a wrong normalisation or gate function.  Each
is a text substitution in a temporary copy of ``oracle/kda_oracle.c``; the committed oracle is
never modified.
"""
import pytest

import oracle
from oracle_pins import PINS

with open(oracle.SOURCE) as _f:
    SRC = _f.read()

DECAY = "for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a;"
R_BLOCK_START = "    /* prediction of the decayed state for key k: r = S'^T k */"
W_BLOCK_START = "    /* delta-rule write: S = S' + beta * k (v - r)^T */"
O_BLOCK_START = "    /* read after the write: o = S^T q */"


def _swap_blocks(src, first, second, end_marker):
    """Move the block starting at `second` (up to `end_marker`) in front of `first`."""
    i1 = src.index(first)
    i2 = src.index(second)
    i3 = src.index(end_marker, i2)
    block = src[i2:i3]
    rest = src[:i2] + src[i3:]
    return rest[:i1] + block + rest[i1:]


MUTANTS = {
    "delta_sign": lambda s: s.replace("(v[j] - r[j])", "(v[j] + r[j])"),
    "no_decay": lambda s: s.replace("double a = exp(clamp_logdecay(g[i]));", "double a = 1.0;"),
    "decay_on_value_axis": lambda s: s.replace(
        DECAY, "for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= exp(clamp_logdecay(g[j % dk]));"),
    "read_before_write": lambda s: _swap_blocks(s, W_BLOCK_START, O_BLOCK_START, "\n}\n"),
    "predict_from_undecayed_state": lambda s: _swap_blocks(
        s, "    /* decay: S'[i][j]", R_BLOCK_START, W_BLOCK_START),
    "no_lower_clamp": lambda s: s.replace("if (g < -5.0) return -5.0;", ""),
    "no_upper_clamp": lambda s: s.replace("if (g > 0.0) return 0.0;", ""),
    "transposed_read": lambda s: s.replace(
        "acc += S[i * dv + j] * q[i];", "acc += S[(j % dk) * dv + (i % dv)] * q[i];"),
    "beta_dropped": lambda s: s.replace(
        "S[i * dv + j] += beta * k[i] * (v[j] - r[j]);", "S[i * dv + j] += k[i] * (v[j] - r[j]);"),
    "prediction_uses_query": lambda s: s.replace(
        "acc += S[i * dv + j] * k[i];", "acc += S[i * dv + j] * q[i];"),
    "chunk_mask_without_diagonal": lambda s: s.replace(
        "for (int64_t s = 0; s <= r; ++s) {", "for (int64_t s = 0; s < r; ++s) {"),
    "chunk_decay_reference_off_by_one": lambda s: s.replace(
        "exp(GC - G[s * dk + i])", "exp(GC - (s > 0 ? G[(s - 1) * dk + i] : 0.0))"),
    # pre-mixer and output gate
    "conv_taps_reversed": lambda s: s.replace(
        "acc += tap[i] * premix_input(", "acc += tap[3 - i] * premix_input("),
    "conv_history_not_reset": lambda s: s.replace(
        "if (t >= start) return x[t * HD + col];", "if (t >= 0) return x[t * HD + col];"),
    "conv_history_rows_reversed": lambda s: s.replace("* 3 + (3 - back)) * HD", "* 3 + (back - 1)) * HD"),
    "norm_without_sqrt": lambda s: s.replace("double nrm = sqrt(ss);", "double nrm = ss;"),
    "norm_over_all_heads": lambda s: s.replace(
        "for (int64_t c = 0; c < d; ++c) ss += y[c] * y[c];",
        "for (int64_t c = 0; c < d; ++c) ss += y[c] * y[c] + y[(c + d) % HD] * y[(c + d) % HD];"),
    "v_normalised_too": lambda s: s.replace("for (int xi = 0; xi < 2; ++xi) {", "for (int xi = 0; xi < 3; ++xi) {"),
    "softplus_sign": lambda s: s.replace("clamp_logdecay(-softplus)", "clamp_logdecay(softplus)"),
    "softplus_without_log": lambda s: s.replace(": log1p(exp(x));", ": exp(x);"),
    "beta_sign": lambda s: s.replace("1.0 / (1.0 + exp(-b[t * n_heads + h]))", "1.0 / (1.0 + exp(b[t * n_heads + h]))"),
    "output_gate_sign": lambda s: s.replace("o[i] / (1.0 + exp(-z[i]))", "o[i] / (1.0 + exp(z[i]))"),
    "output_gate_tanh": lambda s: s.replace("o[i] / (1.0 + exp(-z[i]))", "o[i] * tanh(z[i])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    mutated = MUTANTS[name](SRC)
    assert mutated != SRC, f"mutation {name} did not apply"
    orc = oracle.build_variant(mutated, str(tmp_path))
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake '{name}'"
