"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle source, plants one mistake in the copy (on the CPU,
in a temporary directory), builds it, and runs the pin tests against it: at
least one pin has to fail. The committed oracle is never modified.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "decay dropped": ("S[c * dv + j] *= dec;", "S[c * dv + j] *= 1.0;"),
    "delta sign flipped": ("resid[j] = load_io(t->v, i * t->sv + j, t->io_bf16) - resid[j];",
                           "resid[j] = load_io(t->v, i * t->sv + j, t->io_bf16) + resid[j];"),
    "state read transposed": ("resid[j] += S[c * dv + j] * kn[c];", "resid[j] += S[j * dv + c] * kn[c];"),
    "output reads the key": ("o[j] += S[c * dv + j] * qn[c];", "o[j] += S[c * dv + j] * kn[c];"),
    "q norm without eps": ("double r = 1.0 / sqrt(ss + eps);", "double r = 1.0 / sqrt(ss + 1e-2);"),
    "bwd erase term dropped": ("dSp[c * dv + j] = dS[c * dv + j] - beta * kn[c] * du[j];",
                               "dSp[c * dv + j] = dS[c * dv + j];"),
    "bwd gate grad on dS": ("acc += Spt[c * dv + j] * dSp[c * dv + j];",
                            "acc += Spt[c * dv + j] * dS[c * dv + j];"),
    "bwd norm r^3 term dropped": ("rk * dkn[c] - rk * rk * rk * kr[c] * pk", "rk * dkn[c]"),
    "bwd dv without beta": ("t->dv_[i * t->so + j] = beta * du[j];", "t->dv_[i * t->so + j] = du[j];"),
    "bwd decay not applied to dS": ("dS[c * dv + j] = dec * dSp[c * dv + j];",
                                    "dS[c * dv + j] = dSp[c * dv + j];"),
}


def _pin_calls():
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            calls.append((name, fn, {}))
            continue
        argnames = [a.strip() for a in params[0].args[0].split(",")]
        for vals in params[0].args[1]:
            vals = vals if isinstance(vals, tuple) else (vals,)
            calls.append((name, fn, dict(zip(argnames, vals))))
    return calls


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, "mutation site not found"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"])
    caught = []
    oracle.load(str(so))
    try:
        for name, fn, kw in _pin_calls():
            try:
                fn(**kw) if "tmp_path" not in inspect.signature(fn).parameters else fn(tmp_path=tmp_path, **kw)
            except AssertionError:
                caught.append(name)
            if caught:
                break
    finally:
        oracle.load()
    assert caught, f"no pin caught the mutant '{mutant}'"
