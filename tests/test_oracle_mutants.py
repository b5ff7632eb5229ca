"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/kda_oracle.c``, plants one mistake in the copy
(a dropped term, a wrong sign, a wrong operand or index, a transposed gate, a
read-out taken before the update, a lost token), compiles the copy with gcc
into a temporary folder and runs the independent checks against it. Every
mutant must fail at least one check; the real oracle must pass all of them.
Nothing here touches a GPU.
"""
import json
import os
import re
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import brute

HERE = os.path.dirname(__file__)
SRC = os.path.join(os.path.dirname(HERE), "oracle", "kda_oracle.c")


def _frac(x):
    return np.vectorize(lambda s: float(Fraction(s)))(np.array(x, dtype=object)).astype(np.float64)


def _move_readout_before_update(src: str) -> str:
    start = src.index("        /* o_t = S_t^T q_t */")
    end = src.index("    }\n\n    if (sT)")
    readout = src[start:end]
    src = src[:start] + src[end:]
    at = src.index("        /* S_t = S' + beta_t k_t (v_t - v_hat)^T */")
    return src[:at] + readout + src[at:]


MUTANTS = {
    "prediction_uses_q": ("vhat[j] += S[i * dv + j] * kt[i];", "vhat[j] += S[i * dv + j] * qt[i];"),
    "error_sign": ("(vt[j] - vhat[j])", "(vt[j] + vhat[j])"),
    "gate_dropped": ("S[i * dv + j] *= at[i];", "S[i * dv + j] *= 1.0;"),
    "gate_on_value_axis": ("S[i * dv + j] *= at[i];", "S[i * dv + j] *= at[j % dk];"),
    "beta_dropped": ("const double bk = bt * kt[i];", "const double bk = kt[i];"),
    "readout_uses_k": ("ot[j] += S[i * dv + j] * qt[i];", "ot[j] += S[i * dv + j] * kt[i];"),
    "prediction_wrong_index": ("vhat[j] += S[i * dv + j] * kt[i];",
                               "vhat[j] += S[i * dv + j] * kt[j % dk];"),
    "last_token_lost": ("t < t0 + T; ++t", "t < t0 + T - 1; ++t"),
    "initial_state_ignored": ("    if (s0)\n        memcpy", "    if (0)\n        memcpy"),
    "head_offset_lost_q": ("const double *qt = q + (t * H + h) * dk;",
                           "const double *qt = q + (t * H) * dk;"),
    "beta_wrong_head": ("const double bt = beta[t * H + h];", "const double bt = beta[t * H];"),
    "readout_before_update": (None, _move_readout_before_update),
}


def _battery(lib) -> list[str]:
    """Independent checks; returns the names of the ones that fail."""
    failed = []
    for fname in ("hand_kda_d2x2_t2.json", "hand_kda_d2x3_t1.json"):
        with open(os.path.join(HERE, "golden", fname)) as f:
            g = json.load(f)
        args = [_frac(g[n]) for n in ("q", "k", "v", "alpha", "beta")]
        try:
            o, s = oracle.run(*args, initial_state=_frac(g["initial_state"]), lib=lib)
            if not (np.array_equal(o, _frac(g["expected_o"]))
                    and np.array_equal(s, _frac(g["expected_final_state"]))):
                failed.append(fname)
        except ValueError:
            failed.append(fname)
    rng = np.random.default_rng(0)
    for (dk, dv, T, H) in [(5, 3, 10, 2), (4, 6, 7, 3)]:
        q = rng.standard_normal((2, T, H, dk))
        k = rng.standard_normal((2, T, H, dk))
        v = rng.standard_normal((2, T, H, dv))
        a = rng.uniform(0.05, 1, (2, T, H, dk))
        b = rng.uniform(0, 1, (2, T, H))
        S0 = rng.standard_normal((2, H, dk, dv))
        o, s = oracle.run(q, k, v, a, b, initial_state=S0, lib=lib)
        ob, sb = brute.run(q, k, v, a, b, S0)
        if not (np.allclose(o, ob, atol=1e-12, rtol=0) and np.allclose(s, sb, atol=1e-12, rtol=0)):
            failed.append(f"brute_{dk}x{dv}")
    return failed


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_real_oracle_passes_battery():
    assert _battery(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    if old is None:
        mutated = new(source)
    else:
        assert source.count(old) == 1, f"mutation anchor for {name} not unique"
        mutated = source.replace(old, new)
    assert mutated != source
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    assert _battery(lib), f"planted mistake {name!r} slipped through every pin"
