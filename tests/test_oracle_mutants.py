"""The oracle's pins catch planted mistakes (CPU only).

A pin is only worth something if a wrong oracle fails it.  Each case below
plants one plausible slip in a copy of the oracle -- the C recurrence
(oracle/kda_oracle.c) or the gated RMSNorm (oracle/norm.py) -- by a text
substitution, loads the copy in place of the real one, and runs the pins of
test_oracle.py against it: every mutant must fail at least one.  The slips are
the ones a reader of the recurrence

    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t

could make: a dropped or misplaced decay, the decay on the value axis, a sign,
S k for S^T k, the output read before the write, a lost beta, scale or
initial state, the sigmoid mirrored, an index slip in varlen or verify, and
the norm's eps, mean, weight and gate.  Every planted copy stays in bounds for
the pins' shapes (indices that a slip could push out are wrapped), so a
mutant can fail a pin but cannot fault the process.

The mutants exist only here, in temporary files; the oracle itself is not
changed.
"""
import ctypes
import os
import subprocess
import types

import numpy as np
import pytest

import oracle as oracle_pkg
import test_oracle as pins

C_SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "kda_oracle.c")
NORM_SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "norm.py")

# Pins that take the oracle module, cheapest first.
RECURRENCE_PINS = [
    pins.test_hand_examples,
    pins.test_beta_zero_gate_zero_identity,
    pins.test_beta_zero_pure_decay_closed_form,
    pins.test_scalar_closed_form_with_sigmoid,
    pins.test_retrieval_overwrites_nonzero_state,
    pins.test_exact_retrieval_orthonormal_keys,
    pins.test_matrix_definition_form,
    pins.test_gate_extreme_forgets_state,
    pins.test_linearity_in_values_and_state,
    pins.test_varlen_independence_and_permutation,
    pins.test_continuation_chains_final_to_initial,
    pins.test_verify_matches_prefill_prefixes,
    pins.test_chunked_form_equals_sequential,
]
NORM_PINS = [
    pins.test_gated_rmsnorm_constant_row_closed_form,
    pins.test_gated_rmsnorm_scale_invariance_and_gate_limits,
]

# Step markers of the token update in kda_oracle.c, in their order there.
_DECAY = "    /* decay: S <- Diag(exp g) S */\n"
_READ = "    /* u <- v - S^T k */\n"
_WRITE = "    /* S <- S + beta k u^T */\n"
_OUT = "    /* o <- scale S^T q */\n"
_END = "\n}\n\n/*\n * Prefill"


def _steps(src):
    """Split the token update into (head, decay, read, write, out, tail)."""
    i = [src.index(m) for m in (_DECAY, _READ, _WRITE, _OUT)]
    j = src.index(_END, i[3]) + 1
    return src[:i[0]], src[i[0]:i[1]], src[i[1]:i[2]], src[i[2]:i[3]], src[i[3]:j], src[j:]


def _reorder(order):
    def f(src):
        head, decay, read, write, out, tail = _steps(src)
        parts = dict(decay=decay, read=read, write=write, out=out)
        return head + "".join(parts[p] for p in order) + tail
    return f


def _sub(old, new):
    def f(src):
        assert src.count(old) >= 1, "mutation anchor not found: %r" % old
        return src.replace(old, new, 1)
    return f


C_MUTANTS = {
    "decay dropped": _sub("row[j] *= d;", "row[j] *= 1.0 + 0.0 * d;"),
    "decay sign flipped": _sub("const double d = exp(g[c]);", "const double d = exp(-g[c]);"),
    "decay on the value axis": _sub("for (int64_t j = 0; j < V; ++j) row[j] *= d;",
                                    "for (int64_t j = 0; j < V; ++j) row[j] *= exp(g[j % K]) + 0.0 * d;"),
    "retrieval before the decay": _reorder(["read", "decay", "write", "out"]),
    "decay after the write": _reorder(["read", "write", "decay", "out"]),
    "output before the write": _reorder(["decay", "read", "out", "write"]),
    "delta sign flipped": _sub("u[j] -= row[j] * kc;", "u[j] += row[j] * kc;"),
    "S k instead of S^T k": _sub("for (int64_t j = 0; j < V; ++j) u[j] -= row[j] * kc;",
                                 "for (int64_t j = 0; j < V; ++j) u[j] -= S[(j % K) * V + (c % V)] * kc + 0.0 * row[j];"),
    "beta dropped from the write": _sub("const double bk = beta * k[c];",
                                        "const double bk = k[c] + 0.0 * beta;"),
    "beta sigmoid mirrored": _sub("return 1.0 / (1.0 + exp(-b));", "return 1.0 / (1.0 + exp(b));"),
    "scale dropped": _sub("for (int64_t j = 0; j < V; ++j) o[j] *= scale;",
                          "for (int64_t j = 0; j < V; ++j) o[j] *= 1.0 + 0.0 * scale;"),
    "output queried with k": _sub("const double qc = q[c];", "const double qc = k[c] + 0.0 * q[c];"),
    "initial state ignored": _sub("if (h0)\n", "if (0 && h0)\n"),
    "initial state of another head": _sub("memcpy(S, h0 + ch * K * V,",
                                          "memcpy(S, h0 + (n * H + (H - 1 - h)) * K * V,"),
    "last token of a sequence dropped": _sub("for (int64_t t = cu[n]; t < cu[n + 1]; ++t) {",
                                             "for (int64_t t = cu[n]; t < cu[n + 1] - 1; ++t) {"),
    "verify stores one draft late": _sub("if (t + 1 == accepted[r]) memcpy(dst",
                                         "if (t == accepted[r]) memcpy(dst"),
    "verify ignores the slot": _sub("const int64_t s = slot ? slot[r] : r;",
                                    "const int64_t s = (slot ? 0 : 0) + r;"),
}

NORM_MUTANTS = {
    "eps outside the root": _sub("np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + float(eps))",
                                 "np.sqrt(np.mean(o * o, axis=-1, keepdims=True)) + float(eps)"),
    "sum instead of mean": _sub("np.mean(o * o,", "np.sum(o * o,"),
    "weight dropped": _sub("o / rms * w *", "o / rms *"),
    "gate through silu": _sub("(1.0 / (1.0 + np.exp(-gate)))", "(gate / (1.0 + np.exp(-gate)))"),
    "gate sigmoid mirrored": _sub("np.exp(-gate)", "np.exp(gate)"),
}


def _caught(pin_list, *args):
    for pin in pin_list:
        try:
            pin(*args)
        except Exception:  # an assertion, or a shape error the slip caused
            return pin.__name__
    return None


def test_real_oracle_passes_every_pin():
    """The unmodified oracle passes the same pin list (so a catch below is the
    mutation's doing)."""
    oracle_pkg._load()
    assert _caught(RECURRENCE_PINS, oracle_pkg) is None
    assert _caught(NORM_PINS) is None


@pytest.mark.parametrize("name", sorted(C_MUTANTS))
def test_recurrence_mutant_is_caught(name, tmp_path):
    with open(C_SRC) as f:
        src = C_MUTANTS[name](f.read())
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(c), "-o",
                           str(so), "-lm"])
    oracle_pkg._load()
    saved = oracle_pkg._lib
    oracle_pkg._lib = oracle_pkg._bind(ctypes.CDLL(str(so)))
    try:
        pin = _caught(RECURRENCE_PINS, oracle_pkg)
    finally:
        oracle_pkg._lib = saved
    assert pin is not None, "no pin catches the planted slip: %s" % name


@pytest.mark.parametrize("name", sorted(NORM_MUTANTS))
def test_norm_mutant_is_caught(name, monkeypatch):
    import oracle.norm as norm
    with open(NORM_SRC) as f:
        src = NORM_MUTANTS[name](f.read())
    mod = types.ModuleType("norm_mutant")
    exec(compile(src, "norm_mutant.py", "exec"), mod.__dict__)
    monkeypatch.setattr(norm, "gated_rmsnorm", mod.gated_rmsnorm)
    with np.errstate(all="ignore"):
        pin = _caught(NORM_PINS)
    assert pin is not None, "no pin catches the planted slip: %s" % name
