"""Chunked (chunk-parallel) restatement of KDA in torch fp64 -- test helper.

This is NOT the oracle. It restates the chunk algebra that the CUDA path is
built on, written directly from the gated delta rule of KDA ("Kimi K3 on
Fireworks: Fast RL at frontier scale", training section, KDA paragraph: the
chunk-local work runs in parallel and only a small state passes between chunks).
The tests use it to show that this algebra equals the token-by-token oracle at
several chunk sizes, and its torch autograd serves as an independent backward.

Within a chunk (rows r, j are tokens of the chunk, c a key channel):
    G_r    = sum_{i<=r} g_i                      (per channel, restarts every chunk)
    A_rj   = sum_c k^_rc k^_jc exp(G_rc - G_jc)  (j < r)
    B_rj   = sum_c q^_rc k^_jc exp(G_rc - G_jc)  (j <= r)
    T      = (I + Diag(beta) A)^-1
    U      = T Diag(beta) (V - (K^ * exp G) S)
    O      = (Q^ * exp G) S + B U
    S_next = Diag(exp G_last) S + (K^ * exp(G_last - G))^T U
"""
import torch


def l2n(x, eps, scale=1.0):
    return scale * x / torch.sqrt((x * x).sum(-1, keepdim=True) + eps)


def kda_chunked(q, k, v, beta, g, h0=None, chunk=64, scale=1.0, eps=1e-6):
    """q, k, g: [T, dk]; v: [T, dv]; beta: [T]; h0: [dk, dv]. All fp64. Returns (o, hT)."""
    T, dk = q.shape
    dv = v.shape[1]
    qn, kn = l2n(q, eps, scale), l2n(k, eps)
    S = torch.zeros(dk, dv, dtype=q.dtype) if h0 is None else h0
    outs = []
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        n = e - s
        Q, K, V, b, gg = qn[s:e], kn[s:e], v[s:e], beta[s:e], g[s:e]
        G = torch.cumsum(gg, 0)
        incl = torch.tril(torch.ones(n, n, dtype=torch.bool))
        strict = torch.tril(torch.ones(n, n, dtype=torch.bool), -1)
        diff = (G[:, None, :] - G[None, :, :]).masked_fill(~incl[..., None], 0.0)
        E = torch.exp(diff) * incl[..., None]
        A = torch.einsum("rc,jc,rjc->rj", K, K, E) * strict
        B = torch.einsum("rc,jc,rjc->rj", Q, K, E) * incl
        L = torch.eye(n, dtype=q.dtype) + b[:, None] * A
        Tm = torch.linalg.solve_triangular(L, torch.eye(n, dtype=q.dtype), upper=False,
                                           unitriangular=True)
        gam = torch.exp(G)
        U = Tm @ (b[:, None] * (V - (K * gam) @ S))
        outs.append((Q * gam) @ S + B @ U)
        S = torch.exp(G[-1])[:, None] * S + (K * torch.exp(G[-1] - G)).T @ U
    return torch.cat(outs, 0), S


def kda_token_loop(q, k, v, beta, g, h0=None, scale=1.0, eps=1e-6):
    """Token-by-token loop in torch (differentiable); an independent second oracle."""
    T, dk = q.shape
    dv = v.shape[1]
    S = torch.zeros(dk, dv, dtype=q.dtype) if h0 is None else h0
    qn, kn = l2n(q, eps, scale), l2n(k, eps)
    outs = []
    for t in range(T):
        Sp = torch.exp(g[t])[:, None] * S
        u = beta[t] * (v[t] - Sp.T @ kn[t])
        S = Sp + torch.outer(kn[t], u)
        outs.append(S.T @ qn[t])
    return torch.stack(outs, 0), S
