"""GPU parity of the Attention Residuals kernels against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
TOL = {"bf16": 1e-2, "f32": 1e-4}


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_chunked_gb300 as m
    m.library()
    return m


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def case(T, S, d, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    src = [(torch.randn(T, d, generator=gen) * (0.5 + 0.25 * i)).to(dtype) for i in range(S)]
    w = torch.randn(d, generator=gen) / d ** 0.5
    g = torch.randn(T, d, generator=gen).to(dtype)
    return src, w, g


def check(kda, T, S, d, io, seed, check_dw=True):
    dtype = torch.bfloat16 if io == "bf16" else torch.float32
    src, w, g = case(T, S, d, dtype, seed)
    dsrc = [x.cuda() for x in src]
    out, stats = kda.attnres_fwd(dsrc, w.cuda())
    d_s, dw = kda.attnres_bwd(dsrc, w.cuda(), stats, g.cuda())
    torch.cuda.synchronize()
    o_ref, a_ref, r_ref, l_ref = oracle.attnres_fwd(src, w)
    ds_ref, dw_ref = oracle.attnres_bwd(src, w, g)
    errs = {"out": rel(out.float().cpu(), o_ref), "alpha": rel(stats[0].cpu(), a_ref),
            "rstd": rel(stats[1].cpu(), r_ref), "logit": rel(stats[2].cpu(), l_ref),
            "dsrc": max(rel(d_s[i].float().cpu(), ds_ref[i]) for i in range(S))}
    if check_dw:
        errs["dw"] = rel(dw.cpu(), dw_ref)
    print("attnres", T, S, d, io, {k: f"{v:.2e}" for k, v in errs.items()})
    for k, v in errs.items():
        assert v <= TOL[io], (k, v)


@pytest.mark.parametrize("T,S", [(37, 9), (5, 1), (300, 4)])
def test_attnres_bf16_k3_width(kda, T, S):
    check(kda, T, S, 7168, "bf16", seed=T + S)


def test_attnres_f32(kda):
    check(kda, 20, 3, 256, "f32", seed=9)


@pytest.mark.parametrize("io,d,S", [("f32", 16384, 9), ("bf16", 16384, 9), ("bf16", 8, 2), ("f32", 72, 5)])
def test_attnres_widths(kda, io, d, S):
    # the widest rows (several chunks per thread, one staging buffer), and rows narrower
    # than one chunk per CTA of the cluster
    check(kda, 7, S, d, io, seed=d + S)


def test_attnres_no_tokens(kda):
    src = [torch.empty(0, 64, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    w = torch.randn(64, device="cuda")
    out, stats = kda.attnres_fwd(src, w)
    d_s, dw = kda.attnres_bwd(src, w, stats, torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert out.shape == (0, 64) and torch.all(dw == 0)


def test_attnres_deterministic(kda):
    src, w, g = case(257, 9, 1024, torch.bfloat16, seed=11)
    dsrc = [x.cuda() for x in src]
    r = []
    for _ in range(2):
        out, stats = kda.attnres_fwd(dsrc, w.cuda())
        d_s, dw = kda.attnres_bwd(dsrc, w.cuda(), stats, g.cuda())
        r.append((out, dw, d_s[3]))
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(r[0], r[1]))


def test_attnres_fullsize_sampled(kda):
    # the bench shape (32768 tokens x 9 sources x 7168): sampled tokens against the oracle
    T, S, d = 32768, 9, 7168
    gen = torch.Generator(device="cuda").manual_seed(12)
    src = [torch.randn(T, d, generator=gen, device="cuda").to(torch.bfloat16) for _ in range(S)]
    w = torch.randn(d, generator=gen, device="cuda") / d ** 0.5
    g = torch.randn(T, d, generator=gen, device="cuda").to(torch.bfloat16)
    out, stats = kda.attnres_fwd(src, w)
    d_s, dw = kda.attnres_bwd(src, w, stats, g)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 4095, 20000, T - 1])
    s_rows = [x[rows].cpu() for x in src]
    o_ref, _, _, _ = oracle.attnres_fwd(s_rows, w.cpu())
    ds_ref, _ = oracle.attnres_bwd(s_rows, w.cpu(), g[rows].cpu())
    assert rel(out[rows].float().cpu(), o_ref) <= TOL["bf16"]
    assert max(rel(d_s[i][rows].float().cpu(), ds_ref[i]) for i in range(S)) <= TOL["bf16"]
    assert torch.isfinite(dw).all()
