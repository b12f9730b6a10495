"""Pins for the fp64 oracle: facts fixed by the definition, not by the oracle itself.

Each test checks the oracle against something independent of it: closed forms
of special cases, a hand-worked example, invariants of the recurrence, an
exact-arithmetic finite-difference check of the backward, and an independent
chunked restatement. A plausible slip in the oracle (a dropped term, a wrong
sign, a swapped index or operand) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from chunked_fp64 import kda_chunked, kda_token_loop

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_inputs(T, H, dk, dv, seed, dyadic=False, gmean=3.0):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, dk, generator=gen)
    k = torch.randn(T, H, dk, generator=gen)
    v = torch.randn(T, H, dv, generator=gen)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen))
    g = torch.nn.functional.logsigmoid(torch.randn(T, H, dk, generator=gen) + gmean)
    if dyadic:  # values on a 2^-8 grid so that +-2^-20 perturbations are exact in fp32
        q, k, v, beta, g = [torch.round(x * 256) / 256 for x in (q, k, v, beta, g)]
        beta = beta.clamp(1 / 256, 1.0)
    return q, k, v, beta, g


def cu(*lens):
    return torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)


def run_fwd(q, k, v, beta, g, lens, h0=None, **kw):
    res = oracle.fwd(q, k, v, beta, g, cu(*lens), h0, **kw)
    return oracle.assemble_fwd(res, cu(*lens), q.shape[1], v.shape[2])


def l2n(x, eps=oracle.EPS):
    x = x.double()
    return x / torch.sqrt((x * x).sum(-1, keepdim=True) + eps)


# ---------------------------------------------------------------- closed forms

def test_single_token_closed_form():
    """T=1, zero state: S = beta k^ v^T and o = beta (k^.q^) v."""
    q, k, v, beta, g = rand_inputs(1, 3, 16, 8, seed=1)
    o, hT = run_fwd(q, k, v, beta, g, [1])
    for h in range(3):
        kn, qn = l2n(k[0, h]), l2n(q[0, h])
        S = beta[0, h].double() * torch.outer(kn, v[0, h].double())
        np.testing.assert_allclose(hT[0, h], S.numpy(), rtol=1e-13, atol=1e-15)
        o_ref = beta[0, h].double() * (kn @ qn) * v[0, h].double()
        np.testing.assert_allclose(o[0, h], o_ref.numpy(), rtol=1e-13, atol=1e-15)


def test_worked_example_by_hand():
    rows, hT_ref = [], None
    for line in open(os.path.join(HERE, "golden", "kda_worked_example.txt")):
        line = line.split("#")[0].split()
        if not line:
            continue
        if line[0] == "hT":
            hT_ref = np.array([float(x) for x in line[1:]]).reshape(2, 2)
        else:
            rows.append([float(x) for x in line[1:]])
    R = torch.tensor(rows, dtype=torch.float32)
    k, v, beta, g, q, o_ref = R[:, 0:2], R[:, 2:4], R[:, 4], R[:, 5:7], R[:, 7:9], R[:, 9:11]
    o, hT = run_fwd(q[:, None], k[:, None], v[:, None], beta[:, None], g[:, None], [3], eps=0.0)
    np.testing.assert_allclose(o[:, 0], o_ref.double().numpy(), rtol=0, atol=2e-7)
    np.testing.assert_allclose(hT[0, 0], hT_ref, rtol=0, atol=2e-7)


def test_orthogonal_keys_prefix_sum():
    """g=0, h0=0, mutually orthogonal keys: the erase term vanishes, S_t = sum_{j<=t} beta_j k^_j v_j^T."""
    T, d = 12, 16
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=2)
    perm = torch.randperm(d, generator=torch.Generator().manual_seed(3))[:T]
    k = torch.zeros(T, 1, d)
    for t in range(T):
        k[t, 0, perm[t]] = float(t + 1) * (-1) ** t
    g = torch.zeros_like(g)
    o, hT = run_fwd(q, k, v, beta, g, [T])
    S = torch.zeros(d, d, dtype=torch.float64)
    for t in range(T):
        S = S + beta[t, 0].double() * torch.outer(l2n(k[t, 0]), v[t, 0].double())
        np.testing.assert_allclose(o[t, 0], (S.T @ l2n(q[t, 0])).numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT[0, 0], S.numpy(), rtol=1e-12, atol=1e-14)


def test_orthogonal_keys_beta_one_is_prefix_sum_of_kv():
    T, d = 8, 8
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=4)
    k = torch.eye(d)[:T, None, :] * 2.0
    beta = torch.ones(T, 1)
    g = torch.zeros_like(g)
    o, hT = run_fwd(q, k, v, beta, g, [T], eps=0.0)
    kv = sum(torch.outer(torch.eye(d)[t].double(), v[t, 0].double()) for t in range(T))
    np.testing.assert_allclose(hT[0, 0], kv.numpy(), rtol=1e-12, atol=1e-14)


def test_repeated_unit_key_beta_one_overwrites():
    """beta=1 with one repeated unit key: S_t = k^ v_t^T (the old value is erased)."""
    T, d = 6, 8
    q, _, v, _, g = rand_inputs(T, 1, d, d, seed=5)
    k = torch.zeros(T, 1, d)
    k[:, 0, 3] = 1.0
    h0 = (torch.randn(1, 1, d, d, generator=torch.Generator().manual_seed(6)) * 0.1)
    h0[0, 0, 3, :] = 0.0    # no prior value under this key; other rows must persist
    o, hT = run_fwd(q, k, v, torch.ones(T, 1), torch.zeros_like(g), [T], h0, eps=0.0)
    for t in range(T):
        S = h0[0, 0].double().clone()
        S[3, :] = v[t, 0].double()
        np.testing.assert_allclose(o[t, 0], (S.T @ l2n(q[t, 0], 0.0)).numpy(), rtol=1e-12, atol=1e-14)
    S = h0[0, 0].double().clone()
    S[3, :] = v[-1, 0].double()
    np.testing.assert_allclose(hT[0, 0], S.numpy(), rtol=1e-12, atol=1e-14)


def test_beta_zero_is_pure_decay():
    """beta=0: S_t = Diag(exp(G_t)) h0 with G_t the running sum of g; o_t = S_t^T q^_t."""
    T, d = 9, 16
    q, k, v, _, g = rand_inputs(T, 2, d, d, seed=7)
    h0 = torch.randn(1, 2, d, d, generator=torch.Generator().manual_seed(8))
    o, hT = run_fwd(q, k, v, torch.zeros(T, 2), g, [T], h0)
    for h in range(2):
        G = torch.cumsum(g[:, h].double(), 0)
        for t in range(T):
            S = torch.exp(G[t])[:, None] * h0[0, h].double()
            np.testing.assert_allclose(o[t, h], (S.T @ l2n(q[t, h])).numpy(), rtol=1e-12)
        np.testing.assert_allclose(hT[0, h], (torch.exp(G[-1])[:, None] * h0[0, h].double()).numpy(),
                                   rtol=1e-12)
    # with g = 0 as well, o_t = h0^T q^_t
    o, _ = run_fwd(q, k, v, torch.zeros(T, 2), torch.zeros_like(g), [T], h0)
    for t in range(T):
        np.testing.assert_allclose(o[t, 1], (h0[0, 1].double().T @ l2n(q[t, 1])).numpy(), rtol=1e-12)


def test_forget_gate_reset():
    """g_t = -80 on every channel: the prior state is scaled by exp(-80), S_t ~ beta k^ v^T."""
    T, d = 5, 16
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=9)
    g[2] = -80.0
    h0 = torch.randn(1, 1, d, d, generator=torch.Generator().manual_seed(10))
    o, _ = run_fwd(q, k, v, beta, g, [3], h0)
    kn, qn = l2n(k[2, 0]), l2n(q[2, 0])
    ref = beta[2, 0].double() * (kn @ qn) * v[2, 0].double()
    np.testing.assert_allclose(o[2, 0], ref.numpy(), rtol=1e-9, atol=1e-30)


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunked_form_equals_recurrence(C):
    """The chunk algebra (any chunk size) reproduces the token loop."""
    T, d = 150, 32
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=11)
    h0 = torch.randn(1, 1, d, d, generator=torch.Generator().manual_seed(12)) * 0.1
    o, hT = run_fwd(q, k, v, beta, g, [T], h0)
    oc, Sc = kda_chunked(q[:, 0].double(), k[:, 0].double(), v[:, 0].double(), beta[:, 0].double(),
                         g[:, 0].double(), h0[0, 0].double(), chunk=C)
    np.testing.assert_allclose(o[:, 0], oc.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], Sc.numpy(), rtol=1e-11, atol=1e-12)


def test_chaining_and_varlen_and_heads():
    T1, T2, H, d = 37, 50, 3, 16
    q, k, v, beta, g = rand_inputs(T1 + T2, H, d, d, seed=13)
    o, hT = run_fwd(q, k, v, beta, g, [T1 + T2])
    o1, h1 = run_fwd(q[:T1], k[:T1], v[:T1], beta[:T1], g[:T1], [T1])
    o2, h2 = run_fwd(q[T1:], k[T1:], v[T1:], beta[T1:], g[T1:], [T2],
                     torch.from_numpy(h1).float())
    np.testing.assert_allclose(o[:T1], o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o[T1:], o2, rtol=1e-5, atol=1e-6)   # h1 re-enters as fp32
    np.testing.assert_allclose(hT, h2, rtol=1e-5, atol=1e-6)
    # packed varlen == separate calls
    ov, hv = run_fwd(q, k, v, beta, g, [T1, T2])
    ob, hb = run_fwd(q[T1:], k[T1:], v[T1:], beta[T1:], g[T1:], [T2])
    np.testing.assert_array_equal(ov[:T1], o1)
    np.testing.assert_array_equal(ov[T1:], ob)
    np.testing.assert_array_equal(hv[1], hb[0])
    # permuting heads permutes outputs
    p = [2, 0, 1]
    op, hp = run_fwd(q[:, p], k[:, p], v[:, p], beta[:, p], g[:, p], [T1 + T2])
    np.testing.assert_array_equal(op, o[:, p])
    np.testing.assert_array_equal(hp, hT[:, p])


def test_padding_rows_are_noops():
    """Rows with q=k=v=0, beta=0, g=0 leave the state unchanged and output zero."""
    T, d = 20, 16
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=14)
    o, hT = run_fwd(q, k, v, beta, g, [T])
    ins = [5, 6, 13]
    keep = [i for i in range(T + len(ins))]
    Q, K, V, Bt, G = [torch.zeros(T + len(ins), *x.shape[1:]) for x in (q, k, v, beta, g)]
    src = 0
    real = []
    for i in keep:
        if i in ins:
            continue
        Q[i], K[i], V[i], Bt[i], G[i] = q[src], k[src], v[src], beta[src], g[src]
        real.append(i)
        src += 1
    op, hp = run_fwd(Q, K, V, Bt, G, [T + len(ins)])
    np.testing.assert_allclose(op[real], o, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(op[ins], 0.0)
    np.testing.assert_allclose(hp, hT, rtol=1e-13, atol=1e-15)


def test_decode_equals_forward():
    N, L, H, d = 3, 4, 2, 16
    gen = torch.Generator().manual_seed(15)
    q, k, v = [torch.randn(N, L, H, d, generator=gen) for _ in range(3)]
    beta = torch.sigmoid(torch.randn(N, L, H, generator=gen))
    g = torch.nn.functional.logsigmoid(torch.randn(N, L, H, d, generator=gen) + 3)
    state = torch.randn(N, H, d, d, generator=gen) * 0.02
    acc = torch.tensor([0, 2, 4], dtype=torch.int32)
    res = oracle.step(q, k, v, beta, g, state, acc)
    for i in range(N):
        o_f, _ = run_fwd(q[i], k[i], v[i], beta[i], g[i], [L], state[i:i + 1])
        a = int(acc[i])
        if a:
            _, h_a = run_fwd(q[i, :a], k[i, :a], v[i, :a], beta[i, :a], g[i, :a], [a], state[i:i + 1])
        for h in range(H):
            o_s, s_s = res[(i, h)]
            np.testing.assert_array_equal(o_s, o_f[:, h])
            if a:
                np.testing.assert_array_equal(s_s, h_a[0, h])
            else:
                np.testing.assert_array_equal(s_s, state[i, h].double().numpy())


def test_paged_decode_verify_then_replay():
    # Verify a draft with accept 0 (state untouched), then in one call replay the accepted
    # prefix right-aligned after padding and verify the next draft: the committed state and
    # the new draft's outputs equal the token loop run over the accepted tokens followed by
    # the new draft (the forward recurrence itself, not the decode routine).
    N, L1, L2, H, d = 3, 4, 3, 2, 16
    R = L1
    gen = torch.Generator().manual_seed(21)
    mk = lambda L: ([torch.randn(N, L, H, d, generator=gen) for _ in range(3)],
                    torch.sigmoid(torch.randn(N, L, H, generator=gen)),
                    torch.nn.functional.logsigmoid(torch.randn(N, L, H, d, generator=gen) + 3))
    (q1, k1, v1), b1, g1 = mk(L1)
    (q2, k2, v2), b2, g2 = mk(L2)
    P = 5
    pool = torch.randn(P, H, d, d, generator=gen) * 0.02
    idx = torch.tensor([3, 0, 4], dtype=torch.int32)
    acc = [2, 0, 4]
    # phase 1: verify only
    r1 = oracle.step_paged(q1, k1, v1, b1, g1, pool, idx, [0] * N, [0] * N)
    for i in range(N):
        for h in range(H):
            np.testing.assert_array_equal(r1[(i, h)][1], pool[int(idx[i]), h].double().numpy())
    # phase 2: [pad | accepted prefix | next draft], first_slot = R - a, commit after R slots
    L = R + L2
    cat = lambda a1, a2, zero_shape: torch.stack(
        [torch.cat([torch.zeros(R - acc[i], *zero_shape), a1[i, :acc[i]], a2[i]], 0) for i in range(N)])
    q = cat(q1, q2, (H, d)); k = cat(k1, k2, (H, d)); v = cat(v1, v2, (H, d))
    g = cat(g1, g2, (H, d)); beta = cat(b1, b2, (H,))
    first = [R - a for a in acc]
    r2 = oracle.step_paged(q, k, v, beta, g, pool, idx, first, [R] * N)
    for i in range(N):
        a = acc[i]
        qq = torch.cat([q1[i, :a], q2[i]]); kk = torch.cat([k1[i, :a], k2[i]]); vv = torch.cat([v1[i, :a], v2[i]])
        bb = torch.cat([b1[i, :a], b2[i]]); gg = torch.cat([g1[i, :a], g2[i]])
        s0 = pool[int(idx[i])][None]
        o_f, _ = run_fwd(qq, kk, vv, bb, gg, [a + L2], s0)
        if a:
            _, h_a = run_fwd(qq[:a], kk[:a], vv[:a], bb[:a], gg[:a], [a], s0)
        for h in range(H):
            o_s, s_s = r2[(i, h)]
            np.testing.assert_allclose(o_s, o_f[:, h], rtol=1e-12, atol=1e-14)
            ref = h_a[0, h] if a else pool[int(idx[i]), h].double().numpy()
            np.testing.assert_allclose(s_s, ref, rtol=1e-12, atol=1e-14)


def test_state_map_is_affine():
    # The recurrence is affine in the initial state: the final state from S equals M S + b, with
    # M the final state from the identity with zero values and b the final state from zero.
    T, H, d = 37, 2, 16
    q, k, v, beta, g = rand_inputs(T, H, d, d, seed=61)
    S = torch.randn(1, H, d, d, generator=torch.Generator().manual_seed(62)) * 0.1
    eye = torch.eye(d).expand(1, H, d, d).contiguous()
    _, M = run_fwd(q, k, torch.zeros_like(v), beta, g, [T], eye)
    _, b = run_fwd(q, k, v, beta, g, [T])
    _, hS = run_fwd(q, k, v, beta, g, [T], S)
    for h in range(H):
        np.testing.assert_allclose(hS[0, h], M[0, h] @ S[0, h].double().numpy() + b[0, h], rtol=1e-12, atol=1e-13)


def test_segment_combine_reproduces_unsplit_forward():
    # Context parallelism: cut the sequence into segments, get each segment's (M, b) on its own,
    # chain S_in[k+1] = M[k] S_in[k] + b[k] from h0, rerun every segment from S_in[k]: the outputs
    # and the final state are those of the unsplit forward.
    T, H, d = 100, 2, 16
    q, k, v, beta, g = rand_inputs(T, H, d, d, seed=63)
    h0 = torch.randn(1, H, d, d, generator=torch.Generator().manual_seed(64)) * 0.1
    o_ref, h_ref = run_fwd(q, k, v, beta, g, [T], h0)
    cuts = [0, 30, 64, 81, 100]
    eye = torch.eye(d).expand(1, H, d, d).contiguous()
    s_in = h0[0].double().numpy()
    outs = []
    for a, e in zip(cuts[:-1], cuts[1:]):
        sl = slice(a, e)
        s32 = torch.from_numpy(s_in).float()   # a handed-over state is fp32, as h0 is
        _, M = run_fwd(q[sl], k[sl], torch.zeros_like(v[sl]), beta[sl], g[sl], [e - a], eye)
        _, b = run_fwd(q[sl], k[sl], v[sl], beta[sl], g[sl], [e - a])
        o_seg, h_seg = run_fwd(q[sl], k[sl], v[sl], beta[sl], g[sl], [e - a], s32[None])
        outs.append(o_seg)
        s_next = np.stack([M[0, h] @ s32[h].double().numpy() + b[0, h] for h in range(H)])
        np.testing.assert_allclose(h_seg[0], s_next, rtol=1e-11, atol=1e-12)
        s_in = s_next
    # against the unsplit forward, up to the fp32 rounding of the three handed-over states
    np.testing.assert_allclose(np.concatenate(outs, 0), o_ref, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(s_in, h_ref[0], rtol=1e-5, atol=1e-6)


def test_contraction_bound():
    """|k^|<=1, beta in [0,1], g<=0 make (I - beta k^k^T) Diag(e^g) a contraction:
    |S_t|_F <= |S_{t-1}|_F + beta |v_t|."""
    d = 16
    gen = torch.Generator().manual_seed(16)
    S = torch.randn(1, 1, d, d, generator=gen)
    for t in range(40):
        q, k, v = [torch.randn(1, 1, d, generator=gen) for _ in range(3)]
        beta = torch.rand(1, 1, generator=gen)
        g = -torch.rand(1, 1, d, generator=gen) * 0.3
        _, hT = run_fwd(q, k, v, beta, g, [1], S)
        bound = np.linalg.norm(S[0, 0].double().numpy()) + float(beta) * float(v.double().norm())
        assert np.linalg.norm(hT[0, 0]) <= bound * (1 + 1e-12)
        S = torch.from_numpy(hT).float()


# ------------------------------------------------------------------- backward

def _bwd(q, k, v, beta, g, lens, dO, h0=None, dhT=None, **kw):
    res = oracle.bwd(q, k, v, beta, g, cu(*lens), dO, h0, dhT, **kw)
    return oracle.assemble_bwd(res, cu(*lens), q.shape[1])


@pytest.mark.parametrize("d", [4, 8])
def test_backward_matches_exact_finite_differences(d):
    """Central differences with exactly representable perturbations (dyadic inputs)."""
    T, H = 6, 1
    q, k, v, beta, g = rand_inputs(T, H, d, d, seed=20 + d, dyadic=True)
    gen = torch.Generator().manual_seed(30 + d)
    h0 = torch.round(torch.randn(1, H, d, d, generator=gen) * 64) / 256
    dO = torch.round(torch.randn(T, H, d, generator=gen) * 256) / 256
    dhT = torch.round(torch.randn(1, H, d, d, generator=gen) * 256) / 256
    grads = _bwd(q, k, v, beta, g, [T], dO, h0, dhT)

    def loss(q_, k_, v_, b_, g_, h_):
        o, hT = run_fwd(q_, k_, v_, b_, g_, [T], h_)
        return float((o * dO.double().numpy()).sum() + (hT * dhT.double().numpy()).sum())

    h = 2.0 ** -20
    base = [q, k, v, beta, g, h0]
    names = ["dq", "dk", "dv", "dbeta", "dg", "dh0"]
    for which, name in enumerate(names):
        x = base[which]
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.clone(), x.clone()
            xp[idx] += h
            xm[idx] -= h
            assert float(xp[idx]) - float(xm[idx]) == 2 * h   # perturbation is exact
            ap = list(base); ap[which] = xp
            am = list(base); am[which] = xm
            fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        got = grads[name]
        scale = max(1e-12, np.abs(fd).max())
        assert np.abs(got - fd).max() / scale < 1e-6, name


def test_adjoint_identity():
    """o and hT are jointly linear in (v, h0): <dO,o> + <dhT,hT> = <dv,v> + <dh0,h0>."""
    T, H, d = 70, 2, 16
    q, k, v, beta, g = rand_inputs(T, H, d, d, seed=40)
    gen = torch.Generator().manual_seed(41)
    h0 = torch.randn(1, H, d, d, generator=gen) * 0.1
    dO = torch.randn(T, H, d, generator=gen)
    dhT = torch.randn(1, H, d, d, generator=gen)
    o, hT = run_fwd(q, k, v, beta, g, [T], h0)
    gr = _bwd(q, k, v, beta, g, [T], dO, h0, dhT)
    lhs = (o * dO.double().numpy()).sum() + (hT * dhT.double().numpy()).sum()
    rhs = (gr["dv"] * v.double().numpy()).sum() + (gr["dh0"] * h0.double().numpy()).sum()
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))


@pytest.mark.parametrize("T,d,C", [(20, 8, 4), (130, 32, 64)])
def test_backward_matches_autograd_of_independent_forms(T, d, C):
    """Torch fp64 autograd through an independent token loop and through the chunked form."""
    H = 2
    q, k, v, beta, g = rand_inputs(T, H, d, d, seed=50 + T)
    gen = torch.Generator().manual_seed(51)
    h0 = torch.randn(1, H, d, d, generator=gen) * 0.1
    dO = torch.randn(T, H, d, generator=gen)
    dhT = torch.randn(1, H, d, d, generator=gen)
    gr = _bwd(q, k, v, beta, g, [T], dO, h0, dhT)
    for h in range(H):
        for form in (kda_token_loop, lambda *a: kda_chunked(*a, chunk=C)):
            xs = [x[:, h].double().clone().requires_grad_(True) for x in (q, k, v, beta, g)]
            hh = h0[0, h].double().clone().requires_grad_(True)
            o, S = form(*xs, hh)
            L = (o * dO[:, h].double()).sum() + (S * dhT[0, h].double()).sum()
            L.backward()
            for x, name in zip(xs + [hh], ["dq", "dk", "dv", "dbeta", "dg", "dh0"]):
                ref = x.grad.numpy()
                got = gr[name][0, h] if name == "dh0" else gr[name][:, h]
                np.testing.assert_allclose(got, ref, rtol=1e-9, atol=1e-11 * np.abs(ref).max())


def test_scale_parameter():
    """scale multiplies q^ and hence o (the state is unaffected)."""
    T, d = 10, 16
    q, k, v, beta, g = rand_inputs(T, 1, d, d, seed=60)
    o1, h1 = run_fwd(q, k, v, beta, g, [T])
    o2, h2 = run_fwd(q, k, v, beta, g, [T], scale=0.125)
    np.testing.assert_allclose(o2, 0.125 * o1, rtol=1e-13)
    np.testing.assert_array_equal(h1, h2)
