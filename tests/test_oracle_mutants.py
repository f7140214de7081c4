"""The oracle pins must catch plausible slips.

Each case copies ``oracle/kb_oracle.c`` to a temporary directory, plants one
mistake by text substitution (on the CPU, in the copy only), compiles it and
runs the pin tests against the mutant.  At least one pin has to fail.
"""

import ctypes
import functools
import os
import shutil
import subprocess
import types

import pytest

import oracle
from tests import test_oracle_backward_pins as bwd_pins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kb_oracle.c")

MUTANTS = {
    "dropped_scale": ("scores[j] = dot * inv_sqrt_d;", "scores[j] = dot;"),
    "causal_off_by_one": ("const int ctx = p + 1;", "const int ctx = p + (p > 0 ? 0 : 1);"),
    "gqa_interleaved": ("const int g = h / group;", "const int g = h % J->Hkv;"),
    "wrong_sign": ("scores[j] = exp(scores[j] - m);", "scores[j] = exp(m - scores[j]);"),
    "k_v_swapped": ("const double w = scores[j];\n        for (int d = 0; d < D; ++d) o[d] += w * bf16_to_double(vrow[d]);",
                    "const double w = scores[j];\n        for (int d = 0; d < D; ++d) o[d] += w * bf16_to_double(kbase[(size_t)j * D + d]);"),
    "kv_stride_uses_context": ("((size_t)b * J->Hkv + g) * (size_t)J->cap * D;\n    const uint16_t *vbase",
                               "((size_t)b * J->Hkv + g) * (size_t)ctx * D;\n    const uint16_t *vbase"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) o[d] /= denom;", "(void)denom;"),
}

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_") and n != "test_brute_force_agreement"
             and n != "test_bad_rows_are_rejected"]


def _mutant_module(tmp_path, old, new):
    src = open(SRC).read()
    assert old in src, "mutation anchor not found in the oracle source"
    path = tmp_path / "kb_oracle_mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-pthread", str(path), "-lm", "-o", str(so)],
                   check=True)
    lib = oracle._bind(str(so))
    mod = types.SimpleNamespace(
        attention_rows=functools.partial(oracle.attention_rows, _lib_override=lib),
        attention_full=functools.partial(oracle.attention_full, _lib_override=lib),
        backward=functools.partial(oracle.backward, _lib_override=lib),
        dq_rows=functools.partial(oracle.dq_rows, _lib_override=lib),
    )
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_fails_on_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    mod = _mutant_module(tmp_path, old, new)
    failures = []
    for t in PIN_TESTS + [functools.partial(pins.test_brute_force_agreement, B=1, Hq=8, Hkv=2, S=10, seed=3)]:
        try:
            t(mod)
        except Exception as e:  # noqa: BLE001 - any failure of a pin counts
            failures.append(getattr(t, "__name__", "brute_force"))
    assert failures, f"mutant {name} passed every pin"


# Slips in the gradient code; the forward code of the mutant is untouched, so
# the finite-difference pin compares against a correct forward.
BWD_MUTANTS = {
    "dropped_delta": ("const double ds = p[j] * (dp[j] - delta);", "const double ds = p[j] * dp[j];"),
    "dq_missing_scale": ("dqrow[d] += ds * bf16_to_double(krow[d]) * inv_sqrt_d;",
                         "dqrow[d] += ds * bf16_to_double(krow[d]);"),
    "dk_uses_dout": ("dkrow[d] += ds * qd[d] * inv_sqrt_d;", "dkrow[d] += ds * dod[d] * inv_sqrt_d;"),
    "dv_uses_ds": ("dvrow[d] += p[j] * dod[d];", "dvrow[d] += ds * dod[d];"),
    "delta_unweighted": ("delta += p[j] * dot;", "delta += dot;"),
    "group_interleaved": ("for (int h = g * group; h < (g + 1) * group; ++h) {",
                          "for (int h = g; h < J->Hq; h += J->Hkv) {"),
    "causal_off_by_one": ("softmax_row(qd, kbase, i, D, inv_sqrt_d, p);",
                          "softmax_row(qd, kbase, i > 0 ? i - 1 : 0, D, inv_sqrt_d, p);"),
}

BWD_PIN_TESTS = [getattr(bwd_pins, n) for n in dir(bwd_pins) if n.startswith("test_")]


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_some_backward_pin_fails_on_mutant(tmp_path, name):
    old, new = BWD_MUTANTS[name]
    mod = _mutant_module(tmp_path, old, new)
    failures = []
    for t in BWD_PIN_TESTS:
        try:
            if t is bwd_pins.test_finite_differences:
                t(mod, bwd_pins.make_small_case())
            else:
                t(mod)
        except Exception as e:  # noqa: BLE001 - any failure of a pin counts
            failures.append(t.__name__)
    assert failures, f"mutant {name} passed every backward pin"
