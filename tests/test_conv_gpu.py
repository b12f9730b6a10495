"""GPU parity of the short-convolution kernels (forward, backward, decode step) against the
fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
TOL = {"bf16": 1e-2, "f32": 1e-4}
DT = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def kda():
    import gated_delta_rule_chunked_gb300 as m
    m.library()
    return m


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def case(lens, C, W, io, seed, with_state=True, with_bias=True):
    gen = torch.Generator().manual_seed(seed)
    T, N = sum(lens), len(lens)
    x = torch.randn(T, C, generator=gen).to(DT[io])
    w = torch.randn(C, W, generator=gen) / W ** 0.5
    b = torch.randn(C, generator=gen) * 0.1 if with_bias else None
    st = torch.randn(N, W - 1, C, generator=gen).to(DT[io]) if with_state else None
    dy = torch.randn(T, C, generator=gen).to(DT[io])
    dso = torch.randn(N, W - 1, C, generator=gen)
    cu = torch.tensor(np.cumsum([0] + list(lens)), dtype=torch.int32)
    return x, w, b, st, dy, dso, cu


def cuda(t):
    return None if t is None else t.cuda()


def run_check(kda, lens, C, W, io, act, seed, with_state=True, with_bias=True, with_dso=True, equal=False):
    x, w, b, st, dy, dso, cu = case(lens, C, W, io, seed, with_state, with_bias)
    dso = dso if with_dso else None
    N = len(lens)
    cu_arg = None if equal else cu
    y, so = kda.conv_fwd(x.cuda(), w.cuda(), cuda(b), cuda(cu_arg), cuda(st), activation=act, n_seqs=N)
    g = kda.conv_bwd(x.cuda(), w.cuda(), cuda(b), dy.cuda(), cuda(cu_arg), cuda(st), cuda(dso), activation=act,
                     n_seqs=N)
    torch.cuda.synchronize()
    y_ref, so_ref = oracle.conv_fwd(x, w, b, cu, st, activation=act)
    r = oracle.conv_bwd(x, w, b, cu, st, dy, dso, activation=act)
    errs = {"y": rel(y.float().cpu(), y_ref), "state_out": rel(so.float().cpu(), so_ref),
            "dx": rel(g["dx"].cpu(), r["dx"]), "dweight": rel(g["dweight"].cpu(), r["dweight"]),
            "d_state_in": rel(g["d_state_in"].cpu(), r["d_state_in"])}
    if with_bias:
        errs["dbias"] = rel(g["dbias"].cpu(), r["dbias"])
    print("conv", lens[:6], C, W, io, act, {k: f"{v:.2e}" for k, v in errs.items()})
    for k, v in errs.items():
        assert v <= TOL[io], (k, v)
    # the state after a sequence holds stored inputs: exact
    np.testing.assert_array_equal(so.float().cpu().numpy(), so_ref)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_varlen_ragged(kda, W, io):
    # empty sequences, sequences shorter than W - 1, run-crossing and ragged tails; C spans two CTAs
    lens = [37, 0, 1, 2, 65, 0, 3, 200]
    run_check(kda, lens, 2056, W, io, "silu", seed=W + (10 if io == "f32" else 0))


@pytest.mark.parametrize("act", ["none", "silu"])
def test_conv_no_state_no_bias(kda, act):
    run_check(kda, [100, 31], 512, 4, "bf16", act, seed=5, with_state=False, with_bias=False, with_dso=False)


def test_conv_equal_sequences_without_offsets(kda):
    run_check(kda, [96, 96, 96], 264, 4, "bf16", "silu", seed=6, equal=True)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_long_ranges_varlen(kda, io):
    # wide rows give each CTA a token range of about a hundred rows: whole stages inside a
    # sequence take the backward's plain path, the others the general one
    run_check(kda, [700, 3, 500, 397], 18432, 4, io, "silu", seed=21 if io == "bf16" else 22)


def test_conv_many_short_sequences(kda):
    gen = np.random.default_rng(7)
    lens = [int(v) for v in gen.integers(0, 9, size=150)]
    run_check(kda, lens, 128, 4, "f32", "silu", seed=8)


def test_conv_empty_batch(kda):
    W, C = 4, 64
    st = torch.randn(3, W - 1, C).to(torch.bfloat16).cuda()
    x = torch.empty(0, C, dtype=torch.bfloat16, device="cuda")
    w = torch.randn(C, W).cuda()
    cu = torch.zeros(4, dtype=torch.int32)
    y, so = kda.conv_fwd(x, w, None, cu, st)
    dso = torch.randn(3, W - 1, C).cuda()
    g = kda.conv_bwd(x, w, None, x, cu, st, dso)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(so, st)
    assert torch.equal(g["d_state_in"], dso)
    assert torch.count_nonzero(g["dweight"]) == 0


def test_conv_bwd_is_deterministic(kda):
    x, w, b, st, dy, dso, cu = case([500, 700, 300], 1024, 4, "bf16", seed=9)
    outs = [kda.conv_bwd(x.cuda(), w.cuda(), b.cuda(), dy.cuda(), cu.cuda(), st.cuda(), dso.cuda())
            for _ in range(2)]
    torch.cuda.synchronize()
    for k in ("dx", "dweight", "dbias", "d_state_in"):
        assert torch.equal(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_step_paged_verify_and_padding(kda, io):
    W, C, L, N, P = 4, 2056, 4, 6, 11
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(N, L, C, generator=gen).to(DT[io])
    w = torch.randn(C, W, generator=gen)
    b = torch.randn(C, generator=gen) * 0.1
    pool = torch.randn(P, W - 1, C, generator=gen).to(DT[io])
    idx = torch.tensor([3, 9, 0, 7, 10, 5], dtype=torch.int32)
    first = torch.tensor([0, 1, 0, 3, 4, 2], dtype=torch.int32)
    acc = torch.tensor([4, 0, 2, 4, 4, 1], dtype=torch.int32)
    y_ref, pool_ref = oracle.conv_step(x, w, b, pool, idx, acc, first)
    dpool = pool.cuda()
    y = torch.full((N, L, C), 7.0, dtype=DT[io], device="cuda")   # padding slots must stay untouched
    kda.conv_step(x.cuda(), w.cuda(), b.cuda(), dpool, acc, state_indices=idx, first_slot=first, out=y)
    torch.cuda.synchronize()
    yc = y.float().cpu().numpy()
    mask = ~np.isnan(y_ref)
    assert rel(yc[mask], y_ref[mask]) <= TOL[io]
    assert (yc[~mask] == 7.0).all()
    np.testing.assert_array_equal(dpool.float().cpu().numpy(), pool_ref)


@pytest.mark.parametrize("L,W,C,aligned", [(1, 4, 2056, True), (2, 2, 2056, False), (3, 4, 1032, True),
                                             (5, 4, 1032, False), (7, 2, 3080, True)])
def test_conv_step_slot_counts(kda, L, W, C, aligned):
    """Every register specialisation of the step (slot counts up to 1, 2, 4 and 8) and both
    weight paths (16-byte aligned weight rows read as float4, misaligned ones read per element),
    channel counts that leave the last CTA partly empty, accept lengths 0..L and padding, against
    the oracle."""
    N, P = 9, 13
    gen = torch.Generator().manual_seed(100 + 10 * L + W)
    x = torch.randn(N, L, C, generator=gen).to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen)
    b = torch.randn(C, generator=gen) * 0.1
    pool = torch.randn(P, W - 1, C, generator=gen).to(torch.bfloat16)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    acc = torch.randint(0, L + 1, (N,), generator=gen, dtype=torch.int32)
    first = torch.randint(0, L, (N,), generator=gen, dtype=torch.int32)
    y_ref, pool_ref = oracle.conv_step(x, w, b, pool, idx, acc, first)
    if aligned:
        wd, bd = w.cuda(), b.cuda()
    else:   # weight and bias 4 bytes past a 16-byte boundary
        wbig = torch.zeros(C * W + 1, device="cuda")
        bbig = torch.zeros(C + 1, device="cuda")
        wbig[1:] = w.reshape(-1).cuda()
        bbig[1:] = b.cuda()
        wd, bd = wbig[1:].view(C, W), bbig[1:]
        assert wd.data_ptr() % 16 != 0 and bd.data_ptr() % 16 != 0
    dpool = pool.cuda()
    y = torch.full((N, L, C), 7.0, dtype=torch.bfloat16, device="cuda")
    kda.conv_step(x.cuda(), wd, bd, dpool, acc, state_indices=idx, first_slot=first, out=y)
    torch.cuda.synchronize()
    yc = y.float().cpu().numpy()
    mask = ~np.isnan(y_ref)
    assert rel(yc[mask], y_ref[mask]) <= TOL["bf16"]
    assert (yc[~mask] == 7.0).all()
    np.testing.assert_array_equal(dpool.float().cpu().numpy(), pool_ref)


def test_conv_step_more_than_a_wave(kda):
    """The measured width (C = 3 x 96 x 128) with more CTAs than are resident at once (each
    brings the state and token rows of the CTA one wave later into L2, looking its slot up in
    the pool), one sequence's slot outside the pool: that sequence is reported and untouched,
    the others match the oracle."""
    W, C, L, N, P = 4, 3 * 96 * 128, 4, 24, 32
    gen = torch.Generator().manual_seed(13)
    x = torch.randn(N, L, C, generator=gen).to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen) / 2
    b = torch.randn(C, generator=gen) * 0.1
    pool = torch.randn(P, W - 1, C, generator=gen).to(torch.bfloat16)
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    bad = 9
    idx[bad] = P
    acc = torch.randint(0, L + 1, (N,), generator=gen, dtype=torch.int32)
    first = torch.randint(0, L, (N,), generator=gen, dtype=torch.int32)
    good = [i for i in range(N) if i != bad]
    y_ref, pool_ref = oracle.conv_step(x[good], w, b, pool, idx[good], acc[good], first[good])
    dpool = pool.cuda()
    y = torch.full((N, L, C), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.conv_step(x.cuda(), w.cuda(), b.cuda(), dpool, acc, state_indices=idx, first_slot=first, out=y,
                  dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    yc = y.float().cpu().numpy()
    assert (yc[bad] == 7.0).all()
    yg = yc[good]
    mask = ~np.isnan(y_ref)
    assert rel(yg[mask], y_ref[mask]) <= TOL["bf16"]
    assert (yg[~mask] == 7.0).all()
    np.testing.assert_array_equal(dpool.float().cpu().numpy(), pool_ref)


def test_conv_step_equals_forward(kda):
    W, C, L, N = 3, 512, 8, 5
    gen = torch.Generator().manual_seed(12)
    x = torch.randn(N, L, C, generator=gen).to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen)
    st = torch.randn(N, W - 1, C, generator=gen).to(torch.bfloat16)
    state = st.cuda()
    y = kda.conv_step(x.cuda(), w.cuda(), None, state)
    cu = torch.arange(0, N * L + 1, L, dtype=torch.int32)
    yf, sf = kda.conv_fwd(x.view(N * L, C).cuda(), w.cuda(), None, cu.cuda(), st.cuda())
    torch.cuda.synchronize()
    # one kernel per form, the same arithmetic order per element
    assert torch.equal(y.view(N * L, C), yf)
    assert torch.equal(state, sf)


def test_conv_step_bad_index_reports(kda):
    W, C, N = 4, 64, 2
    x = torch.randn(N, 2, C).to(torch.bfloat16).cuda()
    w = torch.randn(C, W).cuda()
    pool = torch.randn(3, W - 1, C).to(torch.bfloat16).cuda()
    keep = pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.tensor([1, 5], dtype=torch.int32)
    kda.conv_step(x, w, None, pool, state_indices=idx, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.equal(pool[0], keep[0]) and torch.equal(pool[2], keep[2])


def test_conv_fullsize_sampled(kda):
    """The measured workload: q, k, v side by side (C = 3 x 96 x 128), T = 32768, W = 4, SiLU,
    one sequence; sampled rows and channels against the oracle."""
    T, C, W = 32768, 3 * 96 * 128, 4
    gen = torch.Generator(device="cuda").manual_seed(13)
    x = torch.randn(T, C, generator=gen, device="cuda").to(torch.bfloat16)
    dy = torch.randn(T, C, generator=gen, device="cuda").to(torch.bfloat16)
    w = torch.randn(C, W, generator=gen, device="cuda") / 2
    b = torch.randn(C, generator=gen, device="cuda") * 0.1
    st = torch.randn(1, W - 1, C, generator=gen, device="cuda").to(torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    y, so = kda.conv_fwd(x, w, b, cu.cuda(), st)
    g = kda.conv_bwd(x, w, b, dy, cu.cuda(), st, None)
    torch.cuda.synchronize()
    # rows: the start (state rows), run edges, the end; every channel
    xc, dyc, wc, bc, stc = x.cpu(), dy.cpu(), w.cpu(), b.cpu(), st.cpu()
    for t0 in (0, 31, 32, 4095, 16383, T - 5):
        if t0 < W - 1:
            prefix = torch.cat([stc[0, t0:], xc[:t0]], 0) if t0 > 0 else stc[0]
        else:
            prefix = xc[t0 - (W - 1):t0]
        seg = xc[t0:t0 + 4]
        yr, _ = oracle.conv_fwd(seg, wc, bc, torch.tensor([0, seg.shape[0]]), prefix.unsqueeze(0))
        assert rel(y[t0:t0 + 4].float().cpu(), yr) <= TOL["bf16"], t0
    # dweight, dbias and dx over whole columns for a sample of channels
    chans = torch.tensor([0, 1, 7, 8, 4095, 12288, 24575, 36863])
    r = oracle.conv_bwd(xc[:, chans], wc[chans], bc[chans], cu, stc[:, :, chans], dyc[:, chans])
    assert rel(g["dweight"][chans].cpu(), r["dweight"]) <= TOL["bf16"]
    assert rel(g["dbias"][chans].cpu(), r["dbias"]) <= TOL["bf16"]
    assert rel(g["dx"][:, chans].cpu(), r["dx"]) <= TOL["bf16"]
    assert rel(g["d_state_in"][:, :, chans].cpu(), r["d_state_in"]) <= TOL["bf16"]
    np.testing.assert_array_equal(so.float().cpu().numpy(), xc[T - (W - 1):].float().numpy()[None])
