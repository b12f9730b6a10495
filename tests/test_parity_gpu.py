"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Metric per output tensor: max|gpu - oracle| / max|oracle|, at most 1e-2 for
bf16 I/O and 1e-4 for fp32 I/O. The oracle reads exactly the bf16/fp32 values
the GPU reads. Small cases span several chunks with ragged tails; the full-size
workloads are compared on sampled (sequence, head) pairs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_chunked_gb300.inputs import make_seq_batch, make_decode_batch, make_workload, WORKLOADS

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
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all()
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def to_dev(b, dev="cuda"):
    out = {}
    for n in ("q", "k", "v", "beta", "g", "cu_seqlens", "h0", "dO"):
        t = getattr(b, n)
        out[n] = None if t is None else t.to(dev)
    return out


def new_status():
    """A zeroed device status word; kernels write KDA_ERR_TIMEOUT there if a bounded wait gives up."""
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def assert_no_timeout(st):
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())} (a bounded wait gave up)"


def run_fwd(kda, b, save=False, scale=1.0):
    t = to_dev(b)
    st = new_status()
    o, hT, saved = kda.kda_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"],
                               save=save, scale=scale, dev_status=st)
    assert_no_timeout(st)
    return t, o, hT, saved


def check_fwd(kda, b, tol, scale=1.0):
    _, o, hT, _ = run_fwd(kda, b, scale=scale)
    res = oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0, scale=scale)
    o_ref, h_ref = oracle.assemble_fwd(res, b.cu_seqlens, b.heads, 128)
    e_o, e_h = rel(o.float().cpu(), o_ref), rel(hT.cpu(), h_ref)
    print("fwd", f"o {e_o:.2e} hT {e_h:.2e}")
    assert e_o <= tol and e_h <= tol, (e_o, e_h)
    return e_o, e_h


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [129], [200, 1, 64, 130]])
def test_fwd_bf16_ragged(kda, lens):
    b = make_seq_batch(lens, heads=3, io_dtype="bf16", seed=sum(lens), h0=True)
    check_fwd(kda, b, TOL["bf16"])


@pytest.mark.parametrize("lens", [[512], [333, 64]])
def test_fwd_f32(kda, lens):
    b = make_seq_batch(lens, heads=2, io_dtype="f32", seed=len(lens), h0=(len(lens) > 1))
    check_fwd(kda, b, TOL["f32"])


def test_fwd_workload_f32_T512_H2(kda):
    check_fwd(kda, make_workload("fwd-f32-T512-H2"), TOL["f32"])


def test_fwd_zero_state_and_scale(kda):
    b = make_seq_batch([300], heads=2, io_dtype="bf16", seed=5, h0=False)
    check_fwd(kda, b, TOL["bf16"], scale=0.0883883)


def test_fwd_many_heads_selects_wide_slices(kda):
    # n_seqs * heads large enough that the scan uses 64-column value slices
    b = make_seq_batch([70] * 4, heads=96, io_dtype="bf16", seed=11, h0=True)
    check_fwd(kda, b, TOL["bf16"])


def test_fwd_empty_sequences_keep_state(kda):
    b = make_seq_batch([0, 100, 0], heads=2, io_dtype="bf16", seed=12, h0=True)
    _, o, hT, _ = run_fwd(kda, b)
    np.testing.assert_array_equal(hT[0].cpu().numpy(), b.h0[0].numpy())
    np.testing.assert_array_equal(hT[2].cpu().numpy(), b.h0[2].numpy())
    check_fwd(kda, b, TOL["bf16"])


def test_fwd_is_deterministic(kda):
    b = make_seq_batch([400, 77], heads=4, io_dtype="bf16", seed=13, h0=True)
    _, o1, h1, _ = run_fwd(kda, b)
    _, o2, h2, _ = run_fwd(kda, b)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_fwd_chaining_matches_single_call(kda):
    b = make_seq_batch([256], heads=2, io_dtype="bf16", seed=14, h0=True)
    t = to_dev(b)
    o, hT, _ = kda.kda_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], None, t["h0"])
    o1, h1, _ = kda.kda_fwd(t["q"][:128], t["k"][:128], t["v"][:128], t["beta"][:128], t["g"][:128], None, t["h0"])
    o2, h2, _ = kda.kda_fwd(t["q"][128:], t["k"][128:], t["v"][128:], t["beta"][128:], t["g"][128:], None, h1)
    torch.cuda.synchronize()
    assert rel(torch.cat([o1, o2]).float().cpu(), o.float().cpu()) < 1e-2
    assert rel(h2.cpu(), hT.cpu()) < 1e-2


def test_fwd_workload_T4096_H96_full(kda):
    check_fwd(kda, make_workload("fwd-bf16-T4096-H96"), TOL["bf16"])


# ---------------------------------------------------------------- backward

def check_bwd(kda, b, tol, tasks=None):
    t, o, hT, saved = run_fwd(kda, b, save=True)
    gen = torch.Generator().manual_seed(99)
    dhT = (torch.randn(b.n_seqs, b.heads, 128, 128, generator=gen) * 0.1)
    st = new_status()
    gr = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, t["cu_seqlens"], t["h0"],
                     dhT.to("cuda"), dev_status=st)
    assert_no_timeout(st)
    res = oracle.bwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.dO, b.h0, dhT, tasks=tasks)
    errs = {}
    cu = [int(x) for x in b.cu_seqlens.tolist()]
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        gots, refs = [], []
        for (i, h), r in res.items():
            g = gr[name].cpu()
            gots.append((g[i, h] if name == "dh0" else g[cu[i]:cu[i + 1], h]).numpy().ravel())
            refs.append(r[name].ravel())
        errs[name] = rel(np.concatenate(gots), np.concatenate(refs))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    print("bwd", {k: f"{v:.2e}" for k, v in errs.items()})
    assert not bad, errs
    return errs


@pytest.mark.parametrize("lens", [[64], [130], [200, 1, 64, 129]])
def test_bwd_bf16_ragged(kda, lens):
    b = make_seq_batch(lens, heads=3, io_dtype="bf16", seed=100 + sum(lens), h0=True, grad=True)
    check_bwd(kda, b, TOL["bf16"])


@pytest.mark.parametrize("lens", [[64], [130], [200, 1, 64, 129]])
def test_bwd_f32_ragged(kda, lens):
    b = make_seq_batch(lens, heads=2, io_dtype="f32", seed=120 + sum(lens), h0=True, grad=True)
    check_bwd(kda, b, TOL["f32"])


def test_bwd_f32_workload_T512_H2(kda):
    # the fp32 workload's inputs (one 512-token sequence, two heads, zero initial state), dO drawn after them
    check_bwd(kda, make_workload("fwd-f32-T512-H2", kind="fwdbwd"), TOL["f32"])


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_bwd_empty_sequences(kda, io):
    # empty sequences between and around non-empty ones: their dh0 is dhT (nothing to pass back through)
    b = make_seq_batch([0, 70, 0, 65, 0], heads=2, io_dtype=io, seed=115, h0=True, grad=True)
    errs = check_bwd(kda, b, TOL[io])
    assert all(v <= TOL[io] for v in errs.values())


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_bwd_many_heads(kda, io):
    b = make_seq_batch([150, 90], heads=96, io_dtype=io, seed=101, h0=True, grad=True)
    check_bwd(kda, b, TOL[io], tasks=[(0, 0), (0, 57), (1, 95)])


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_bwd_zero_state_no_dhT_scaled(kda, io):
    # h0 = 0 (not passed), no final-state gradient, q scale != 1: dh0 is still the gradient at h0 = 0
    b = make_seq_batch([130, 64, 1], heads=2, io_dtype=io, seed=113, h0=False, grad=True)
    assert b.h0 is None
    t = to_dev(b)
    sc = 128 ** -0.5
    o, hT, saved = kda.kda_fwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], None, save=True, scale=sc)
    gr = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, t["cu_seqlens"], None, None,
                     scale=sc)
    torch.cuda.synchronize()
    res = oracle.bwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.dO, None, None, scale=sc)
    cu = [int(x) for x in b.cu_seqlens.tolist()]
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        got, ref = [], []
        for (i, h), r in res.items():
            g_ = gr[name].cpu()
            got.append((g_[i, h] if name == "dh0" else g_[cu[i]:cu[i + 1], h]).numpy().ravel())
            ref.append(r[name].ravel())
        e = rel(np.concatenate(got), np.concatenate(ref))
        assert e <= TOL[io], (name, e)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_bwd_is_deterministic(kda, io):
    b = make_seq_batch([300], heads=2, io_dtype=io, seed=102, h0=True, grad=True)
    t, o, hT, saved = run_fwd(kda, b, save=True)
    g1 = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, None, t["h0"])
    g2 = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, None, t["h0"])
    for name in g1:
        assert torch.equal(g1[name], g2[name]), name


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_bwd_into_caller_buffers(kda, io):
    # out= writes the same gradients into the caller's tensors (reused across calls); the tensors
    # start as NaN, so a kernel that read an output before writing it would show (the fp32 path
    # keeps intermediates in dq, dk and dg between its two chunk kernels)
    b = make_seq_batch([300, 77], heads=2, io_dtype=io, seed=103, h0=True, grad=True)
    t, o, hT, saved = run_fwd(kda, b, save=True)
    g1 = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, t["cu_seqlens"], t["h0"])
    out = {n: torch.full_like(v, float("nan")) for n, v in g1.items() if v is not None}
    g2 = kda.kda_bwd(t["q"], t["k"], t["v"], t["beta"], t["g"], t["dO"], saved, t["cu_seqlens"], t["h0"], out=out)
    for name in out:
        assert g2[name].data_ptr() == out[name].data_ptr(), name
        assert torch.equal(g1[name], out[name]), name


def _strong_gates(b, kind, seed):
    """Replace the batch's log-decay with gates at the documented bound (every g >= -5)."""
    gen = torch.Generator().manual_seed(seed)
    if kind == "const":        # every 16-token sub-block sums to exactly -80 on every channel
        b.g = torch.full_like(b.g, -5.0)
    elif kind == "uniform":    # g ~ U[-5, 0]
        b.g = -5.0 * torch.rand(b.g.shape, generator=gen, dtype=torch.float32)
    else:                      # channels alternate between the bound and a slow decay
        g = torch.full_like(b.g, -5.0)
        g[..., 1::2] = -0.01
        b.g = g
    return b


@pytest.mark.parametrize("kind", ["const", "uniform", "mixed"])
def test_fwd_gates_at_bound_bf16(kda, kind):
    b = _strong_gates(make_seq_batch([200, 1, 64, 130], heads=3, io_dtype="bf16", seed=110, h0=True), kind, 7)
    check_fwd(kda, b, TOL["bf16"])


@pytest.mark.parametrize("kind", ["const", "mixed"])
def test_fwd_gates_at_bound_f32(kda, kind):
    b = _strong_gates(make_seq_batch([333, 64], heads=2, io_dtype="f32", seed=111, h0=True), kind, 8)
    check_fwd(kda, b, TOL["f32"])


@pytest.mark.parametrize("kind", ["const", "uniform", "mixed"])
def test_bwd_gates_at_bound_bf16(kda, kind):
    b = _strong_gates(make_seq_batch([200, 1, 64, 129], heads=3, io_dtype="bf16", seed=112, h0=True, grad=True),
                      kind, 9)
    check_bwd(kda, b, TOL["bf16"])


@pytest.mark.parametrize("kind", ["const", "uniform", "mixed"])
def test_bwd_gates_at_bound_f32(kda, kind):
    b = _strong_gates(make_seq_batch([333, 64], heads=2, io_dtype="f32", seed=114, h0=True, grad=True), kind, 11)
    check_bwd(kda, b, TOL["f32"])


# ---------------------------------------------------------------- decode

def check_step(kda, d, tol):
    dev = "cuda"
    st = d.state.to(dev)
    o = kda.kda_step(d.q.to(dev), d.k.to(dev), d.v.to(dev), d.beta.to(dev), d.g.to(dev), st,
                     d.accept_len.to(dev))
    torch.cuda.synchronize()
    N, L, H, _ = d.q.shape
    res = oracle.step(d.q, d.k, d.v, d.beta, d.g, d.state, d.accept_len)
    o_ref = np.stack([np.stack([res[(i, h)][0] for h in range(H)], 1) for i in range(N)])
    s_ref = np.stack([np.stack([res[(i, h)][1] for h in range(H)], 0) for i in range(N)])
    e_o, e_s = rel(o.float().cpu(), o_ref), rel(st.cpu(), s_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s)


@pytest.mark.parametrize("N,L", [(5, 4), (3, 1), (2, 8)])
def test_step_bf16(kda, N, L):
    check_step(kda, make_decode_batch(N, L, 3, "bf16", seed=N * 10 + L), TOL["bf16"])


def test_step_f32(kda):
    check_step(kda, make_decode_batch(4, 4, 2, "f32", seed=3), TOL["f32"])


def test_step_gates_at_bound(kda):
    # decode applies exp(g) token by token: strong decay needs no factoring, checked anyway
    d = make_decode_batch(4, 4, 3, "bf16", seed=6)
    gen = torch.Generator().manual_seed(60)
    d.g = -5.0 * torch.rand(d.g.shape, generator=gen, dtype=torch.float32)
    d.g[1] = -5.0
    check_step(kda, d, TOL["bf16"])


def test_step_accept_zero_leaves_state(kda):
    d = make_decode_batch(3, 4, 2, "bf16", seed=4)
    d.accept_len[:] = torch.tensor([0, 4, 0], dtype=torch.int32)
    st = d.state.clone().cuda()
    kda.kda_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.beta.cuda(), d.g.cuda(), st, d.accept_len.cuda())
    torch.cuda.synchronize()
    assert torch.equal(st[0].cpu(), d.state[0]) and torch.equal(st[2].cpu(), d.state[2])
    check_step(kda, d, TOL["bf16"])


def test_step_equals_forward(kda):
    d = make_decode_batch(2, 4, 2, "bf16", seed=5)
    d.accept_len[:] = 4
    st = d.state.clone().cuda()
    o = kda.kda_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.beta.cuda(), d.g.cuda(), st)
    for i in range(2):
        of, hf, _ = kda.kda_fwd(d.q[i].cuda(), d.k[i].cuda(), d.v[i].cuda(), d.beta[i].cuda(), d.g[i].cuda(),
                                None, d.state[i:i + 1].cuda())
        torch.cuda.synchronize()
        assert rel(o[i].float().cpu(), of.float().cpu()) < 1e-2
        assert rel(st[i].cpu(), hf[0].cpu()) < 1e-2


def _paged_case(N, L, H, P, seed):
    d = make_decode_batch(N, L, H, "bf16", seed=seed)
    gen = torch.Generator().manual_seed(seed + 7)
    pool = torch.randn(P, H, 128, 128, generator=gen) * 0.02
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    first = torch.randint(0, L + 1, (N,), generator=gen, dtype=torch.int32)
    acc = torch.randint(0, L + 1, (N,), generator=gen, dtype=torch.int32)
    return d, pool, idx, first, acc


def check_paged(kda, d, pool, idx, first, acc):
    N, L, H, _ = d.q.shape
    st = pool.clone().cuda()
    o = torch.full(d.v.shape, 7.0, dtype=d.v.dtype, device="cuda")   # padded slots keep this
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.beta.cuda(), d.g.cuda(), st, acc.cuda(), out=o,
                 state_indices=idx.cuda(), first_slot=first.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    res = oracle.step_paged(d.q, d.k, d.v, d.beta, d.g, pool, idx.tolist(), first.tolist(), acc.tolist())
    o, st = o.float().cpu(), st.cpu()
    touched = set()
    for i in range(N):
        f, slot = int(first[i]), int(idx[i])
        touched.add(slot)
        assert torch.all(o[i, :f] == 7.0), i
        for h in range(H):
            o_ref, s_ref = res[(i, h)]
            if f < L:
                assert rel(o[i, f:, h], o_ref) <= TOL["bf16"], (i, h)
            assert rel(st[slot, h], s_ref) <= TOL["bf16"], (i, h)
    for slot in range(pool.shape[0]):
        if slot not in touched:
            assert torch.equal(st[slot], pool[slot]), slot


def test_step_paged_pool(kda):
    check_paged(kda, *_paged_case(6, 4, 3, 11, seed=31))


def test_step_paged_full_padding_and_eight_slots(kda):
    d, pool, idx, first, acc = _paged_case(5, 8, 2, 9, seed=32)
    first[0], acc[0] = 8, 8       # all padding: nothing written, state unchanged
    first[1], acc[1] = 3, 2       # commit point inside the padding: state unchanged
    check_paged(kda, d, pool, idx, first, acc)


def test_step_verify_then_replay(kda):
    # phase 1 verifies a draft without committing; phase 2 replays the accepted prefix and
    # verifies the next draft in one call (padding first): committed states and the new draft's
    # outputs match the oracle's token loop over accepted prefix + new draft
    N, L1, L2, H, P = 4, 4, 4, 2, 6
    d1 = make_decode_batch(N, L1, H, "bf16", seed=41)
    d2 = make_decode_batch(N, L2, H, "bf16", seed=42)
    gen = torch.Generator().manual_seed(43)
    pool = torch.randn(P, H, 128, 128, generator=gen) * 0.02
    idx = torch.tensor([5, 1, 2, 0], dtype=torch.int32)
    acc = torch.tensor([3, 0, 4, 1], dtype=torch.int32)
    st = pool.clone().cuda()
    zeros = torch.zeros(N, dtype=torch.int32, device="cuda")
    kda.kda_step(d1.q.cuda(), d1.k.cuda(), d1.v.cuda(), d1.beta.cuda(), d1.g.cuda(), st, zeros,
                 state_indices=idx.cuda())
    torch.cuda.synchronize()
    assert torch.equal(st.cpu(), pool)
    R = L1
    cat = lambda a1, a2: torch.stack([torch.cat([torch.zeros_like(a1[i, :R - int(acc[i])]), a1[i, :int(acc[i])],
                                                 a2[i]], 0) for i in range(N)])
    q, k, v = cat(d1.q, d2.q), cat(d1.k, d2.k), cat(d1.v, d2.v)
    beta, g = cat(d1.beta, d2.beta), cat(d1.g, d2.g)
    first = (R - acc).to(torch.int32)
    o = kda.kda_step(q.cuda(), k.cuda(), v.cuda(), beta.cuda(), g.cuda(), st, torch.full((N,), R, dtype=torch.int32),
                     state_indices=idx.cuda(), first_slot=first.cuda())
    torch.cuda.synchronize()
    for i in range(N):
        a = int(acc[i])
        qq = torch.cat([d1.q[i, :a], d2.q[i]])[None]; kk = torch.cat([d1.k[i, :a], d2.k[i]])[None]
        vv = torch.cat([d1.v[i, :a], d2.v[i]])[None]; bb = torch.cat([d1.beta[i, :a], d2.beta[i]])[None]
        gg = torch.cat([d1.g[i, :a], d2.g[i]])[None]
        slot = int(idx[i])
        res = oracle.step(qq, kk, vv, bb, gg, pool[slot:slot + 1], torch.tensor([a], dtype=torch.int32))
        for h in range(H):
            o_ref, s_ref = res[(0, h)]
            assert rel(o[i, R:, h].float().cpu(), o_ref[a:]) <= TOL["bf16"], (i, h)
            assert rel(st[slot, h].cpu(), s_ref) <= TOL["bf16"], (i, h)


def test_step_bad_state_index_reports(kda):
    d, pool, idx, first, acc = _paged_case(3, 4, 2, 4, seed=51)
    idx[1] = 4                     # outside the pool of 4 slots
    st = pool.clone().cuda()
    o = torch.full(d.v.shape, 7.0, dtype=d.v.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.beta.cuda(), d.g.cuda(), st, acc.cuda(), out=o,
                 state_indices=idx.cuda(), first_slot=first.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1                      # KDA_ERR_INVALID_ARG
    assert torch.all(o[1].float() == 7.0)               # that sequence is left untouched


def test_step_paged_more_than_a_wave(kda):
    """More CTAs than are resident at once (each brings the state of the CTA one wave later
    into L2, looking its slot up in the pool), with one sequence's slot outside the pool: that
    sequence is reported and left untouched, sampled (sequence, head) pairs of the others match
    the oracle, and pool slots no sequence addresses are unchanged."""
    N, L, H, P = 40, 4, 96, 64
    d = make_decode_batch(N, L, H, "bf16", seed=61)
    gen = torch.Generator().manual_seed(68)
    pool = torch.randn(P, H, 128, 128, generator=gen) * 0.02
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    bad = 17
    idx[bad] = P + 3
    first = torch.randint(0, L, (N,), generator=gen, dtype=torch.int32)
    acc = torch.randint(1, L + 1, (N,), generator=gen, dtype=torch.int32)
    st = pool.cuda()
    o = torch.full(d.v.shape, 7.0, dtype=d.v.dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_step(d.q.cuda(), d.k.cuda(), d.v.cuda(), d.beta.cuda(), d.g.cuda(), st, acc.cuda(), out=o,
                 state_indices=idx.cuda(), first_slot=first.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1                      # KDA_ERR_INVALID_ARG
    assert torch.all(o[bad].float() == 7.0)
    seqs, heads = [0, 5, 16, 18, 29, 39], [0, 47, 95]
    sub = lambda t: t[seqs][:, :, heads]
    res = oracle.step_paged(sub(d.q), sub(d.k), sub(d.v), sub(d.beta), sub(d.g), pool[:, heads],
                            [int(idx[i]) for i in seqs], [int(first[i]) for i in seqs], [int(acc[i]) for i in seqs])
    oc, stc = o.float().cpu(), st.cpu()
    for a, i in enumerate(seqs):
        f, slot = int(first[i]), int(idx[i])
        for b, h in enumerate(heads):
            o_ref, s_ref = res[(a, b)]
            assert rel(oc[i, f:, h], o_ref) <= TOL["bf16"], (i, h)
            assert rel(stc[slot, h], s_ref) <= TOL["bf16"], (i, h)
    used = {int(x) for x in idx.tolist()}
    for slot in range(P):
        if slot not in used:
            assert torch.equal(stc[slot], pool[slot]), slot


# ---------------------------------------------------------------- context parallelism (emulated)

def test_cp_combine_vs_fp64_chain(kda):
    N, P, H = 2, 3, 2
    gen = torch.Generator().manual_seed(71)
    M = torch.randn(N, P, H, 128, 128, generator=gen) / 12
    b = torch.randn(N, P, H, 128, 128, generator=gen) * 0.1
    h0 = torch.randn(N, H, 128, 128, generator=gen) * 0.1
    s_in = kda.kda_cp_combine(M.cuda(), b.cuda(), h0.cuda(), P).cpu()
    for n in range(N):
        for h in range(H):
            s = h0[n, h].double()
            for kk in range(P):
                assert rel(s_in[n, kk, h], s.numpy()) <= 1e-5, (n, kk, h)
                s = M[n, kk, h].double() @ s + b[n, kk, h].double()


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_fwd_identity_start_zero_values(kda, io):
    # the segment map: final state from the identity with zero values, no outputs written
    b = make_seq_batch([300, 64], heads=2, io_dtype=io, seed=72, h0=False)
    t = to_dev(b)
    M, _ = kda._fwd_states(t["q"], t["k"], None, t["beta"], t["g"], t["cu_seqlens"], None, 2, scale=1.0,
                           h0_identity=True)
    eye = torch.eye(128).expand(2, 2, 128, 128).contiguous()
    res = oracle.fwd(b.q, b.k, torch.zeros_like(b.v), b.beta, b.g, b.cu_seqlens, eye)
    _, m_ref = oracle.assemble_fwd(res, b.cu_seqlens, 2, 128)
    assert rel(M.cpu(), m_ref) <= TOL[io]


@pytest.mark.parametrize("lens,P,io", [([1000], 3, "bf16"), ([1000], 1, "bf16"), ([100, 900], 4, "bf16"),
                                       ([1000], 3, "f32"), ([100, 900], 4, "f32")])
def test_fwd_cp_matches_unsplit(kda, lens, P, io):
    b = make_seq_batch(lens, heads=3, io_dtype=io, seed=73 + P, h0=True)
    t = to_dev(b)
    o, hT = kda.kda_fwd_cp(t["q"], t["k"], t["v"], t["beta"], t["g"], b.cu_seqlens.cpu(), t["h0"], n_segments=P)
    res = oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0)
    o_ref, h_ref = oracle.assemble_fwd(res, b.cu_seqlens, 3, 128)
    e_o, e_h = rel(o.float().cpu(), o_ref), rel(hT.cpu(), h_ref)
    print("cp", lens, P, io, f"o {e_o:.2e} hT {e_h:.2e}")
    assert e_o <= TOL[io] and e_h <= TOL[io], (e_o, e_h)


def test_fwd_cp_equal_sequences_without_offsets_and_no_h0(kda):
    # cu_seqlens = NULL (two equal sequences), zero initial state, 5 segments of a 640-token
    # sequence (10 chunks: segments of 2 chunks each); bit-identical to a second call
    b = make_seq_batch([640, 640], heads=2, io_dtype="bf16", seed=75)
    t = to_dev(b)
    o, hT = kda.kda_fwd_cp(t["q"], t["k"], t["v"], t["beta"], t["g"], None, None, n_segments=5, n_seqs=2)
    o2, hT2 = kda.kda_fwd_cp(t["q"], t["k"], t["v"], t["beta"], t["g"], None, None, n_segments=5, n_seqs=2)
    res = oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, None)
    o_ref, h_ref = oracle.assemble_fwd(res, b.cu_seqlens, 2, 128)
    e_o, e_h = rel(o.float().cpu(), o_ref), rel(hT.cpu(), h_ref)
    assert e_o <= TOL["bf16"] and e_h <= TOL["bf16"], (e_o, e_h)
    assert torch.equal(o, o2) and torch.equal(hT, hT2)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_fwd_cp_gates_at_bound(kda, io):
    # the segment maps M of strongly decaying segments are tiny (entries underflow): the
    # chained states must still match the unsplit forward
    b = _strong_gates(make_seq_batch([700, 300], heads=2, io_dtype=io, seed=74, h0=True), "uniform", 10)
    t = to_dev(b)
    o, hT = kda.kda_fwd_cp(t["q"], t["k"], t["v"], t["beta"], t["g"], b.cu_seqlens.cpu(), t["h0"], n_segments=4)
    res = oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0)
    o_ref, h_ref = oracle.assemble_fwd(res, b.cu_seqlens, 2, 128)
    e_o, e_h = rel(o.float().cpu(), o_ref), rel(hT.cpu(), h_ref)
    assert e_o <= TOL[io] and e_h <= TOL[io], (e_o, e_h)


# ---------------------------------------------------------------- full-size workloads (sampled)

def _sampled(b, heads):
    """CPU copies of the inputs restricted to the sampled heads (all tokens)."""
    from gated_delta_rule_chunked_gb300.inputs import SeqBatch
    pick = lambda t: None if t is None else t[:, heads].cpu()
    return SeqBatch(pick(b.q), pick(b.k), pick(b.v), pick(b.beta), pick(b.g), b.cu_seqlens.cpu(),
                    None if b.h0 is None else b.h0[:, heads].cpu(), pick(b.dO))


@pytest.mark.parametrize("name,tasks", [
    # six heads spread over the 96 (first, last and middle ones: different CTAs of every kernel)
    ("fwdbwd-bf16-T32768-H96", [(0, 0), (0, 19), (0, 38), (0, 57), (0, 76), (0, 95)]),
    # one head in each of the eight packed sequences, first to last head
    ("fwdbwd-bf16-varlen8-T131072-H96", [(0, 1), (1, 13), (2, 27), (3, 40), (4, 55), (5, 68), (6, 81), (7, 94)]),
])
def test_fullsize_fwd_bwd_sampled(kda, name, tasks):
    dev = torch.device("cuda")
    b = make_workload(name, device=dev)
    heads = sorted({h for _, h in tasks})
    st = new_status()
    o, hT, saved = kda.kda_fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0, save=True, dev_status=st)
    gr = kda.kda_bwd(b.q, b.k, b.v, b.beta, b.g, b.dO, saved, b.cu_seqlens, b.h0, dev_status=st)
    assert_no_timeout(st)
    s = _sampled(b, heads)
    cu = [int(x) for x in b.cu_seqlens.tolist()]
    otasks = [(i, heads.index(h)) for i, h in tasks]
    fres = oracle.fwd(s.q, s.k, s.v, s.beta, s.g, s.cu_seqlens, s.h0, tasks=otasks)
    bres = oracle.bwd(s.q, s.k, s.v, s.beta, s.g, s.cu_seqlens, s.dO, s.h0, tasks=otasks)
    errs = {}
    for (i, h), (i2, hh) in zip(tasks, otasks):
        sl = slice(cu[i], cu[i + 1])
        pairs = {"o": (o[sl, h].float().cpu(), fres[(i2, hh)][0]), "hT": (hT[i, h].cpu(), fres[(i2, hh)][1])}
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            pairs[n] = (gr[n][sl, h].cpu(), bres[(i2, hh)][n])
        pairs["dh0"] = (gr["dh0"][i, h].cpu(), bres[(i2, hh)]["dh0"])
        for n, (g_, r_) in pairs.items():
            errs[f"{n}[{i},{h}]"] = rel(g_, r_)
    bad = {k: v for k, v in errs.items() if not v <= TOL["bf16"]}
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    worst = max(errs, key=errs.get)
    print(f"{name}: largest error {worst} = {errs[worst]:.2e} (tolerance {TOL['bf16']:.0e})")
    assert not bad, errs


def test_fullsize_decode_sampled(kda):
    dev = torch.device("cuda")
    d = make_workload("decode-bf16-N256-L4-H96", device=dev)
    st = d.state.clone()
    o = kda.kda_step(d.q, d.k, d.v, d.beta, d.g, st, d.accept_len)
    torch.cuda.synchronize()
    seqs = [0, 17, 128, 255]
    heads = [0, 33, 95]
    sub = lambda t: t[seqs][:, :, heads].cpu() if t.dim() >= 3 else t[seqs].cpu()
    res = oracle.step(sub(d.q), sub(d.k), sub(d.v), sub(d.beta), sub(d.g), d.state[seqs][:, heads].cpu(),
                      d.accept_len[seqs].cpu())
    go = np.stack([[o[i, :, h].float().cpu().numpy() for h in heads] for i in seqs])
    ro = np.stack([[res[(a, b_)][0] for b_ in range(len(heads))] for a in range(len(seqs))])
    gs = np.stack([[st[i, h].cpu().numpy() for h in heads] for i in seqs])
    rs = np.stack([[res[(a, b_)][1] for b_ in range(len(heads))] for a in range(len(seqs))])
    print("decode-bf16-N256-L4-H96", f"o {rel(go, ro):.2e} state {rel(gs, rs):.2e}")
    assert rel(go, ro) <= TOL["bf16"] and rel(gs, rs) <= TOL["bf16"], (rel(go, ro), rel(gs, rs))
