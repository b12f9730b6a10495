"""CPU pins of the Attention Residuals oracle: closed forms, invariants, and the backward
against torch fp64 autograd of an independent forward and against central differences."""
import numpy as np
import torch

import oracle


def rand_sources(T, S, d, seed):
    gen = torch.Generator().manual_seed(seed)
    src = [torch.randn(T, d, generator=gen) * (1 + i) for i in range(S)]
    w = torch.randn(d, generator=gen) / d ** 0.5
    return src, w


def test_identical_sources_return_the_source():
    x = torch.randn(5, 32, generator=torch.Generator().manual_seed(1))
    w = torch.randn(32, generator=torch.Generator().manual_seed(2))
    out, alpha, _, _ = oracle.attnres_fwd([x, x, x], w)
    np.testing.assert_allclose(out, x.double().numpy(), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(alpha, 1 / 3, rtol=1e-14)


def test_zero_query_averages():
    src, _ = rand_sources(4, 5, 16, seed=3)
    out, alpha, _, _ = oracle.attnres_fwd(src, torch.zeros(16))
    np.testing.assert_allclose(alpha, 0.2, rtol=1e-14)
    np.testing.assert_allclose(out, torch.stack(src).double().mean(0).numpy(), rtol=1e-13, atol=1e-14)


def test_scale_invariance_of_the_scores():
    # RMS normalisation: scaling one source leaves every score unchanged (eps aside)
    src, w = rand_sources(3, 4, 64, seed=4)
    _, a1, _, l1 = oracle.attnres_fwd(src, w, eps=1e-30)
    src2 = list(src)
    src2[2] = src2[2] * 8.0   # exact in fp32
    _, a2, _, l2 = oracle.attnres_fwd(src2, w, eps=1e-30)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)
    np.testing.assert_allclose(a1.sum(-1), 1.0, rtol=1e-14)


def test_backward_matches_autograd_of_an_independent_forward():
    T, S, d = 6, 9, 40
    src, w = rand_sources(T, S, d, seed=5)
    g = torch.randn(T, d, generator=torch.Generator().manual_seed(6))
    ds, dw = oracle.attnres_bwd(src, w, g)
    xs = [x.double().clone().requires_grad_(True) for x in src]
    wd = w.double().clone().requires_grad_(True)
    # the same map written per source, without the stacked form the oracle uses
    scores = torch.stack([(wd * (x / torch.sqrt((x * x).mean(-1, keepdim=True) + oracle.EPS))).sum(-1) for x in xs], -1)
    a = torch.exp(scores - scores.max(-1, keepdim=True).values)
    a = a / a.sum(-1, keepdim=True)
    out = sum(a[:, i:i + 1] * xs[i] for i in range(S))
    (out * g.double()).sum().backward()
    for i in range(S):
        np.testing.assert_allclose(ds[i], xs[i].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw, wd.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_central_differences():
    T, S, d = 2, 3, 8
    src, w = rand_sources(T, S, d, seed=7)
    g = torch.randn(T, d, generator=torch.Generator().manual_seed(8)).double()
    ds, dw = oracle.attnres_bwd(src, w, g)
    loss = lambda s_, w_: float((torch.from_numpy(oracle.attnres_fwd(s_, w_)[0]) * g).sum())
    h = 1e-6
    for i in range(S):
        for t, c in ((0, 1), (1, 5)):
            sp = [x.double().clone() for x in src]
            sm = [x.double().clone() for x in src]
            sp[i][t, c] += h
            sm[i][t, c] -= h
            np.testing.assert_allclose((loss(sp, w.double()) - loss(sm, w.double())) / (2 * h), ds[i][t, c],
                                       rtol=1e-6, atol=1e-8)
    for c in (0, 7):
        wp, wm = w.double().clone(), w.double().clone()
        wp[c] += h
        wm[c] -= h
        np.testing.assert_allclose((loss(src, wp) - loss(src, wm)) / (2 * h), dw[c], rtol=1e-6, atol=1e-8)


def test_constant_source_closed_form():
    # x = c everywhere: RMS = |c| (up to eps), so r = (c^2 + eps)^(-1/2) and logit = r c sum(w)
    d, eps = 16, 1e-6
    w = torch.linspace(-1.0, 2.0, d)
    src = [torch.full((1, d), 3.0), torch.full((1, d), -0.5)]
    _, alpha, rstd, logit = oracle.attnres_fwd(src, w, eps=eps)
    r = np.array([(9.0 + eps) ** -0.5, (0.25 + eps) ** -0.5])
    np.testing.assert_allclose(rstd[0], r, rtol=1e-14)
    np.testing.assert_allclose(logit[0], r * np.array([3.0, -0.5]) * float(w.double().sum()), rtol=1e-13)
    e = np.exp(logit[0] - logit[0].max())
    np.testing.assert_allclose(alpha[0], e / e.sum(), rtol=1e-14)
