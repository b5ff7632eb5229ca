"""The gradient oracle's pins must catch plausible mistakes.

Each case copies ``oracle/kda_oracle_bwd.c``, plants one mistake (a wrong
sign, a dropped factor, a state from the wrong step, a term accumulated in
the wrong order, a replay started from the wrong checkpoint, an ignored
input), compiles the copy with gcc into a temporary folder and runs the
finite-difference and closed-form checks against it. Every mutant must fail
at least one; the real file passes them all. Nothing here touches a GPU.
"""
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(__file__)
SRC = os.path.join(os.path.dirname(HERE), "oracle", "kda_oracle_bwd.c")

MUTANTS = {
    "dk_sign": ("dkk[th * dk + i] = bt * (ge - sw);", "dkk[th * dk + i] = bt * (ge + sw);"),
    "dk_missing_prediction_term": ("dkk[th * dk + i] = bt * (ge - sw);", "dkk[th * dk + i] = bt * ge;"),
    "dv_missing_beta": ("dvv[th * dv + j] = bt * w[j];", "dvv[th * dv + j] = w[j];"),
    "dbeta_uses_v_not_error": ("db += w[j] * e[j];", "db += w[j] * vt[j];"),
    "dalpha_uses_new_state": ("da += g * Sprev[i * dv + j];", "da += g * Scur[i * dv + j];"),
    "gate_left_out_of_chain": ("G[i * dv + j] = at[i] * dSp[i * dv + j];", "G[i * dv + j] = dSp[i * dv + j];"),
    "erase_term_dropped": ("const double g = G[i * dv + j] - bt * kt[i] * w[j];",
                           "const double g = G[i * dv + j];"),
    "dq_from_previous_state": ("s += Scur[i * dv + j] * dot[j];", "s += Sprev[i * dv + j] * dot[j];"),
    "final_state_gradient_ignored": ("    if (dsT)\n        memcpy(G, dsT", "    if (0)\n        memcpy(G, dsT"),
    "replay_from_wrong_checkpoint": ("memcpy(seg, ck + (size_t)c * SZ, SZ * sizeof(double));",
                                     "memcpy(seg, ck + (size_t)(c > 0 ? c - 1 : 0) * SZ, SZ * sizeof(double));"),
    "readout_gradient_after_prediction": (None, "move_readout"),
}


def _move_readout(src: str) -> str:
    """Add q do^T into G only after w = G^T k was formed."""
    start = src.index("            /* G += q_t do_t^T */")
    end = src.index("            /* dq_t = S_t do_t */")
    block = src[start:end]
    src = src[:start] + src[end:]
    at = src.index("            /* dv_t, dbeta_t */")
    return src[:at] + block + src[at:]


def _battery(lib) -> list[str]:
    import test_oracle_backward_pins as P
    failed = []
    checks = {
        "fd_small": lambda: P._fd_check(P._inputs(1, 9, 1, 4, 3, seed=11), _g(lib, P._inputs(1, 9, 1, 4, 3, seed=11)),
                                        coords=25),
        "fd_two_stretches": lambda: P._fd_check(P._inputs(1, 70, 1, 4, 3, seed=12),
                                                _g(lib, P._inputs(1, 70, 1, 4, 3, seed=12)), coords=25),
        "frozen_state": lambda: _frozen(lib),
    }
    for name, fn in checks.items():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def _g(lib, x):
    return oracle.backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["do"], x["dsT"],
                           initial_state=x["S0"], lib=lib)


def _frozen(lib):
    import test_oracle_backward_pins as P
    x = P._inputs(1, 5, 1, 4, 3, seed=13)
    x["alpha"][:] = 1.0
    x["beta"][:] = 0.0
    g = _g(lib, x)
    S0, dS = x["S0"][0, 0], x["dsT"][0, 0]
    q, do = x["q"][0, :, 0], x["do"][0, :, 0]
    np.testing.assert_allclose(g["dq"][0, :, 0], do @ S0.T, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(g["d_initial_state"][0, 0], dS + q.T @ do, rtol=1e-12, atol=1e-13)


def _compile(tmp_path, src_text, name):
    src = tmp_path / f"{name}.c"
    src.write_text(src_text)
    out = str(tmp_path / f"lib{name}.so")
    oracle.build(force=True, src=str(src), out=out)
    return oracle.load_backward(out)


def test_real_gradient_oracle_passes_the_battery(tmp_path):
    lib = _compile(tmp_path, open(SRC).read(), "real")
    assert _battery(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    text = open(SRC).read()
    old, new = MUTANTS[name]
    if old is None:
        mutated = _move_readout(text)
    else:
        assert text.count(old) == 1, f"mutation site of {name} not unique"
        mutated = text.replace(old, new)
    assert mutated != text
    lib = _compile(tmp_path, mutated, name)
    assert _battery(lib), f"mutant {name} passed every check"
