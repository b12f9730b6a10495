"""CPU pins of the short-convolution oracle: the library's grouped conv1d, closed forms
(identity and shift filters), state chaining, the backward against fp64 autograd of an
independent conv1d forward and against central differences, and decode against the forward."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def rand_case(T, C, W, seed, N=1):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, C, generator=gen)
    w = torch.randn(C, W, generator=gen) / W ** 0.5
    b = torch.randn(C, generator=gen) * 0.1
    st = torch.randn(N, W - 1, C, generator=gen)
    return x, w, b, st


def conv1d_ref(x, w, b, prefix, activation):
    """Causal depthwise conv through torch's grouped conv1d over [prefix; x] (fp64)."""
    C, W = w.shape
    xs = torch.cat([prefix, x], 0).T.unsqueeze(0)                 # [1, C, W-1+T]
    z = F.conv1d(xs, w.unsqueeze(1), b, groups=C)[0].T             # valid outputs: T rows
    return F.silu(z) if activation == "silu" else z


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("activation", ["none", "silu"])
def test_matches_grouped_conv1d(W, activation):
    x, w, b, st = rand_case(37, 24, W, seed=10 + W)
    cu = torch.tensor([0, 37])
    y0, _ = oracle.conv_fwd(x, w, b, cu, None, activation=activation)
    ref0 = conv1d_ref(x.double(), w.double(), b.double(), torch.zeros(W - 1, 24, dtype=torch.float64), activation)
    np.testing.assert_allclose(y0, ref0.numpy(), rtol=1e-13, atol=1e-13)
    y1, s1 = oracle.conv_fwd(x, w, None, cu, st, activation=activation)
    ref1 = conv1d_ref(x.double(), w.double(), None, st[0].double(), activation)
    np.testing.assert_allclose(y1, ref1.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(s1[0], x[37 - (W - 1):].double().numpy())


def test_identity_and_shift_filters():
    W, C = 4, 16
    x, _, _, st = rand_case(9, C, W, seed=3)
    cu = torch.tensor([0, 9])
    ident = torch.zeros(C, W)
    ident[:, W - 1] = 1.0
    y, _ = oracle.conv_fwd(x, ident, None, cu, st, activation="none")
    np.testing.assert_array_equal(y, x.double().numpy())
    shift = torch.zeros(C, W)
    shift[:, 0] = 1.0                                              # y[t] = x[t - (W - 1)]
    y, _ = oracle.conv_fwd(x, shift, None, cu, st, activation="none")
    np.testing.assert_array_equal(y[W - 1:], x[:9 - (W - 1)].double().numpy())
    np.testing.assert_array_equal(y[:W - 1], st[0].double().numpy())


@pytest.mark.parametrize("T1", [0, 1, 2, 5, 20])
def test_chaining_through_the_state(T1):
    W, C, T = 4, 12, 20
    x, w, b, st = rand_case(T, C, W, seed=40 + T1)
    y, s = oracle.conv_fwd(x, w, b, torch.tensor([0, T]), st)
    ya, sa = oracle.conv_fwd(x[:T1], w, b, torch.tensor([0, T1]), st)
    yb, sb = oracle.conv_fwd(x[T1:], w, b, torch.tensor([0, T - T1]), torch.from_numpy(sa).float())
    np.testing.assert_allclose(np.concatenate([ya, yb]), y, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(sb, s)


def test_varlen_equals_separate_calls_and_short_sequences_keep_state():
    W, C = 4, 8
    lens = [5, 0, 1, 2, 9]
    cu = torch.tensor(np.cumsum([0] + lens))
    x, w, b, st = rand_case(sum(lens), C, W, seed=7, N=len(lens))
    y, s = oracle.conv_fwd(x, w, b, cu, st)
    for n, L in enumerate(lens):
        s0 = int(cu[n])
        yn, sn = oracle.conv_fwd(x[s0:s0 + L], w, b, torch.tensor([0, L]), st[n:n + 1])
        np.testing.assert_array_equal(y[s0:s0 + L], yn)
        np.testing.assert_array_equal(s[n], sn[0])
    # a sequence of length 1 shifts the state by one row; length 0 keeps it
    np.testing.assert_array_equal(s[1], st[1].double().numpy())
    np.testing.assert_array_equal(s[2], np.concatenate([st[2, 1:].double().numpy(), x[5:6].double().numpy()]))


def _autograd(x, w, b, cu, st, dy, dso, activation):
    xs, ws, bs, ss = (t.double().clone().requires_grad_(True) for t in (x, w, b, st))
    loss = 0.0
    for n in range(cu.numel() - 1):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        if s1 > s0:
            yn = conv1d_ref(xs[s0:s1], ws, bs, ss[n], activation)
            loss = loss + (yn * dy[s0:s1].double()).sum()
        full = torch.cat([ss[n], xs[s0:s1]], 0)
        son = full[full.shape[0] - (w.shape[1] - 1):]
        loss = loss + (son * dso[n].double()).sum()
    loss.backward()
    return xs.grad, ws.grad, bs.grad, ss.grad


@pytest.mark.parametrize("activation", ["none", "silu"])
@pytest.mark.parametrize("W", [2, 4])
def test_backward_matches_autograd_of_conv1d(activation, W):
    lens = [7, 1, 0, 12]
    cu = torch.tensor(np.cumsum([0] + lens))
    C = 10
    x, w, b, st = rand_case(sum(lens), C, W, seed=60 + W, N=len(lens))
    gen = torch.Generator().manual_seed(61)
    dy = torch.randn(sum(lens), C, generator=gen)
    dso = torch.randn(len(lens), W - 1, C, generator=gen)
    r = oracle.conv_bwd(x, w, b, cu, st, dy, dso, activation=activation)
    gx, gw, gb, gs = _autograd(x, w, b, cu, st, dy, dso, activation)
    np.testing.assert_allclose(r["dx"], gx.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dweight"], gw.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["dbias"], gb.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["d_state_in"], gs.numpy(), rtol=1e-12, atol=1e-12)


def test_backward_central_differences():
    W, C = 3, 3
    lens = [4, 1]
    cu = torch.tensor(np.cumsum([0] + lens))
    x, w, b, st = (t.double() for t in rand_case(sum(lens), C, W, seed=80, N=2))
    gen = torch.Generator().manual_seed(81)
    dy = torch.randn(sum(lens), C, generator=gen, dtype=torch.float64)
    dso = torch.randn(2, W - 1, C, generator=gen, dtype=torch.float64)

    def loss(x_, w_, b_, s_):
        y, so = oracle.conv_fwd(x_, w_, b_, cu, s_)
        return float((y * dy.numpy()).sum() + (so * dso.numpy()).sum())

    r = oracle.conv_bwd(x, w, b, cu, st, dy, dso)
    h = 1e-6
    for name, t, key in (("x", x, "dx"), ("w", w, "dweight"), ("b", b, "dbias"), ("s", st, "d_state_in")):
        num = np.zeros(t.shape)
        for idx in np.ndindex(*t.shape):
            tp, tm = t.clone(), t.clone()
            tp[idx] += h
            tm[idx] -= h
            args_p = {"x": x, "w": w, "b": b, "s": st}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            num[idx] = (loss(args_p["x"], args_p["w"], args_p["b"], args_p["s"]) -
                        loss(args_m["x"], args_m["w"], args_m["b"], args_m["s"])) / (2 * h)
        np.testing.assert_allclose(r[key], num, rtol=1e-6, atol=1e-8)


def test_step_equals_forward_with_padding_and_accept():
    W, C, L = 4, 16, 6
    N, P = 4, 7
    gen = torch.Generator().manual_seed(90)
    x = torch.randn(N, L, C, generator=gen)
    w = torch.randn(C, W, generator=gen)
    b = torch.randn(C, generator=gen)
    pool = torch.randn(P, W - 1, C, generator=gen)
    idx = torch.tensor([5, 0, 3, 6])
    first = torch.tensor([0, 2, 5, 1])
    acc = torch.tensor([6, 1, 6, 3])
    y, new_pool = oracle.conv_step(x, w, b, pool, idx, acc, first)
    for n in range(N):
        Fs, a, slot = int(first[n]), int(acc[n]), int(idx[n])
        yf, _ = oracle.conv_fwd(x[n, Fs:], w, b, torch.tensor([0, L - Fs]), pool[slot:slot + 1])
        np.testing.assert_allclose(y[n, Fs:], yf, rtol=1e-14, atol=1e-14)
        assert np.isnan(y[n, :Fs]).all()
        if a > Fs:
            _, sf = oracle.conv_fwd(x[n, Fs:a], w, b, torch.tensor([0, a - Fs]), pool[slot:slot + 1])
            np.testing.assert_array_equal(new_pool[slot], sf[0])
        else:
            np.testing.assert_array_equal(new_pool[slot], pool[slot].double().numpy())
    for slot in (1, 2, 4):   # slots no sequence addresses
        np.testing.assert_array_equal(new_pool[slot], pool[slot].double().numpy())
