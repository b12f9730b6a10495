"""The pins of the torch-written oracle functions (short convolution, Attention
Residuals) must catch plausible mistakes.

Each case takes one oracle function's source, plants one mistake in a copy, swaps the
copy in for the duration of the case, and runs that function family's pin tests: at
least one pin has to fail. The committed oracle is never modified.
"""
import inspect
import textwrap

import pytest

import oracle
import test_attnres_oracle as attnres_pins
import test_conv_oracle as conv_pins

MUTANTS = {
    ("conv_fwd", "tap order reversed"): ("z += Wt[:, j] * xs[j:j + L]", "z += Wt[:, W - 1 - j] * xs[j:j + L]"),
    ("conv_fwd", "state rows reversed"): ("xs = torch.cat([prev, X[s0:s1]], 0)",
                                          "xs = torch.cat([prev.flip(0), X[s0:s1]], 0)"),
    ("conv_fwd", "bias dropped"): ("else bias.double().expand(L, C).clone()", "else 0.0 * bias.double().expand(L, C)"),
    ("conv_fwd", "state after one row late"): ("state_out[n] = xs[xs.shape[0] - (W - 1):]",
                                               "state_out[n] = xs[xs.shape[0] - W:xs.shape[0] - 1]"),
    ("conv_fwd", "SiLU dropped"): ("y[s0:s1] = _conv_act(z, activation)", "y[s0:s1] = z"),
    ("conv_bwd", "SiLU derivative without its z term"): ("dz = G[s0:s1] * sg * (1.0 + z * (1.0 - sg))",
                                                         "dz = G[s0:s1] * sg"),
    ("conv_bwd", "state-out gradient ignored"): ("dxs[xs.shape[0] - (W - 1):] += d_state_out[n].double()",
                                                 "dxs[xs.shape[0] - (W - 1):] += 0.0 * d_state_out[n].double()"),
    ("conv_bwd", "dweight taps mirrored"): ("dW[:, j] += (dz * xs[j:j + L]).sum(0)",
                                            "dW[:, W - 1 - j] += (dz * xs[j:j + L]).sum(0)"),
    ("conv_bwd", "input gradient one row early"): ("dxs[j:j + L] += Wt[:, j] * dz", "dxs[j:j + L] += Wt[:, j - 1] * dz"),
    ("conv_step", "commits one slot late"): ("kept = xs[:W - 1 + a - F]", "kept = xs[:W + a - F]"),
    ("conv_step", "padding slots read"): ("xs = torch.cat([pool[slot].double(), X[n, F:]], 0)",
                                          "xs = torch.cat([pool[slot].double(), X[n, :L - F]], 0)"),
    ("attnres_fwd", "RMS as a sum"): ("rstd = (X.pow(2).mean(-1) + eps).rsqrt()", "rstd = (X.pow(2).sum(-1) + eps).rsqrt()"),
    ("attnres_fwd", "softmax over tokens"): ("alpha = torch.softmax(logit, -1)", "alpha = torch.softmax(logit, 0)"),
    ("attnres_fwd", "scores without the norm"): ("logit = rstd * (X @ wd)", "logit = X @ wd"),
    ("attnres_bwd", "RMS-norm projection dropped"): (
        "dX = dX + rstd.unsqueeze(-1) * (dN - N * (dN * N).sum(-1, keepdim=True) / d)",
        "dX = dX + rstd.unsqueeze(-1) * dN"),
    ("attnres_bwd", "softmax Jacobian mean dropped"): (
        "dlogit = alpha * (dalpha - (alpha * dalpha).sum(-1, keepdim=True))", "dlogit = alpha * dalpha"),
    ("attnres_bwd", "dw from raw sources"): ("dw = (dlogit.unsqueeze(-1) * N).sum((0, 1))",
                                             "dw = (dlogit.unsqueeze(-1) * X).sum((0, 1))"),
}
FAMILY = {"conv_fwd": conv_pins, "conv_bwd": conv_pins, "conv_step": conv_pins,
          "attnres_fwd": attnres_pins, "attnres_bwd": attnres_pins}


def _pin_calls(mod):
    calls = []
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        grid = [{}]
        for m in params:
            argnames = [a.strip() for a in m.args[0].split(",")]
            grid = [dict(g, **dict(zip(argnames, v if isinstance(v, tuple) else (v,)))) for g in grid for v in m.args[1]]
        calls += [(name, fn, kw) for kw in grid]
    return calls


@pytest.mark.parametrize("key", sorted(MUTANTS), ids=lambda k: f"{k[0]}: {k[1]}")
def test_pins_catch_planted_mistake(key):
    fname, _ = key
    old, new = MUTANTS[key]
    original = getattr(oracle, fname)
    src = textwrap.dedent(inspect.getsource(original))
    assert src.count(old) == 1, "mutation site not found"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), f"<mutant of {fname}>", "exec"), ns)
    caught = []
    setattr(oracle, fname, ns[fname])
    try:
        for name, fn, kw in _pin_calls(FAMILY[fname]):
            try:
                fn(**kw)
            except Exception:   # a failed assertion, or the mistake breaking the computation
                caught.append(name)
                break
    finally:
        setattr(oracle, fname, original)
    assert caught, f"no pin caught the mutant {key}"


@pytest.mark.parametrize("fname", sorted(FAMILY))
def test_unmodified_copies_pass_every_pin(fname):
    # the control: a copy made the same way, without a mistake, is caught by nothing
    original = getattr(oracle, fname)
    ns = dict(vars(oracle))
    exec(compile(textwrap.dedent(inspect.getsource(original)), f"<copy of {fname}>", "exec"), ns)
    setattr(oracle, fname, ns[fname])
    try:
        for name, fn, kw in _pin_calls(FAMILY[fname]):
            fn(**kw)
    finally:
        setattr(oracle, fname, original)
