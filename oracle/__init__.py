"""fp64 CPU oracle for Kimi Delta Attention -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline arm
may import this package. It shares no code with the CUDA library: the arithmetic
is the plain token-by-token loop in ``kda_oracle.c`` (see its header for the
definition and the passages it follows), loaded here through ctypes.

Inputs are torch CPU tensors in their stored dtype (bf16 or fp32); the C code
widens them exactly to double. Outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Iterable, Optional

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_oracle.c")
LIB = os.path.join(HERE, "libkda_oracle.so")
EPS = 1e-6


class Task(C.Structure):
    _fields_ = [
        ("T", C.c_int64), ("dk", C.c_int32), ("dv", C.c_int32), ("io_bf16", C.c_int32),
        ("scale", C.c_double), ("eps", C.c_double),
        ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("dO", C.c_void_p),
        ("sq", C.c_int64), ("sk", C.c_int64), ("sv", C.c_int64), ("sdo", C.c_int64),
        ("beta", C.c_void_p), ("sbeta", C.c_int64),
        ("g", C.c_void_p), ("sg", C.c_int64),
        ("h0", C.c_void_p), ("dhT", C.c_void_p),
        ("accept", C.c_int64),
        ("so", C.c_int64), ("sb", C.c_int64),
        ("o", C.c_void_p), ("hT", C.c_void_p),
        ("dq", C.c_void_p), ("dk_", C.c_void_p), ("dv_", C.c_void_p), ("dg", C.c_void_p),
        ("dbeta", C.c_void_p), ("dh0", C.c_void_p),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP). Returns the library path."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


_lib = None


def load(path: Optional[str] = None):
    """Load the oracle library (default: build and load ``libkda_oracle.so``).

    The mutation tests pass the path of a deliberately broken copy to check
    that the pins catch it; ``load()`` switches back to the real one.
    """
    global _lib
    if path is None:
        path = build()
    handle = C.CDLL(path)
    for fn in ("kda_oracle_fwd", "kda_oracle_bwd", "kda_oracle_step"):
        getattr(handle, fn).argtypes = [C.POINTER(Task), C.c_int, C.c_int]
        getattr(handle, fn).restype = None
    _lib = handle
    return handle


def lib():
    return _lib if _lib is not None else load()


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def _host(t: Optional[torch.Tensor]):
    """A contiguous CPU view of an input, keeping bf16 bit patterns as int16."""
    if t is None:
        return None, False
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16), True
    if t.dtype != torch.float32:
        t = t.to(torch.float32)
    return t, False


def _ptr(t: Optional[torch.Tensor], offset_elems: int = 0):
    if t is None:
        return None
    return t.data_ptr() + offset_elems * t.element_size()


class _Prepared:
    def __init__(self, q, k, v, beta, g, cu_seqlens, h0, dO, dhT):
        self.q, bf = _host(q)
        self.k, _ = _host(k)
        self.v, _ = _host(v)
        self.dO, _ = _host(dO)
        self.bf16 = bf
        self.beta, _ = _host(beta)
        self.g, _ = _host(g)
        self.h0, _ = _host(h0)
        self.dhT, _ = _host(dhT)
        self.cu = [int(x) for x in cu_seqlens.to("cpu").tolist()]
        self.H = self.q.shape[1]
        self.dk = self.q.shape[2]
        self.dv = self.v.shape[2]


def _task(P: _Prepared, i: int, h: int, scale: float, eps: float) -> Task:
    t0, t1 = P.cu[i], P.cu[i + 1]
    H, dk, dv = P.H, P.dk, P.dv
    st = Task()
    st.T = t1 - t0
    st.dk, st.dv, st.io_bf16 = dk, dv, int(P.bf16)
    st.scale, st.eps = scale, eps
    st.q = _ptr(P.q, (t0 * H + h) * dk)
    st.k = _ptr(P.k, (t0 * H + h) * dk)
    st.v = _ptr(P.v, (t0 * H + h) * dv)
    st.dO = _ptr(P.dO, (t0 * H + h) * dv) if P.dO is not None else None
    st.sq = st.sk = H * dk
    st.sv = st.sdo = H * dv
    st.beta = _ptr(P.beta, t0 * H + h)
    st.sbeta = H
    st.g = _ptr(P.g, (t0 * H + h) * dk)
    st.sg = H * dk
    st.h0 = _ptr(P.h0, (i * H + h) * dk * dv) if P.h0 is not None else None
    st.dhT = _ptr(P.dhT, (i * H + h) * dk * dv) if P.dhT is not None else None
    return st


def _all_tasks(P: _Prepared):
    return [(i, h) for i in range(len(P.cu) - 1) for h in range(P.H)]


def fwd(q, k, v, beta, g, cu_seqlens, h0=None, *, scale: float = 1.0, eps: float = EPS,
        tasks: Optional[Iterable] = None, n_threads: int = 0):
    """Forward for the given (sequence, head) tasks (default: all).

    Returns ``{(i, h): (o [T_i, dv], hT [dk, dv])}`` as float64 arrays.
    """
    P = _Prepared(q, k, v, beta, g, cu_seqlens, h0, None, None)
    tasks = list(tasks) if tasks is not None else _all_tasks(P)
    arr = (Task * max(1, len(tasks)))()
    out = {}
    for n, (i, h) in enumerate(tasks):
        st = _task(P, i, h, scale, eps)
        o = np.zeros((st.T, P.dv), np.float64)
        hT = np.zeros((P.dk, P.dv), np.float64)
        st.o, st.hT, st.so = o.ctypes.data, hT.ctypes.data, P.dv
        arr[n] = st
        out[(i, h)] = (o, hT)
    lib().kda_oracle_fwd(arr, len(tasks), n_threads or default_threads())
    return out


def bwd(q, k, v, beta, g, cu_seqlens, dO, h0=None, dhT=None, *, scale: float = 1.0,
        eps: float = EPS, tasks: Optional[Iterable] = None, n_threads: int = 0):
    """Backward for the given tasks. Returns ``{(i, h): dict(dq, dk, dv, dg, dbeta, dh0)}``."""
    P = _Prepared(q, k, v, beta, g, cu_seqlens, h0, dO, dhT)
    tasks = list(tasks) if tasks is not None else _all_tasks(P)
    arr = (Task * max(1, len(tasks)))()
    out = {}
    for n, (i, h) in enumerate(tasks):
        st = _task(P, i, h, scale, eps)
        r = {"dq": np.zeros((st.T, P.dk)), "dk": np.zeros((st.T, P.dk)),
             "dv": np.zeros((st.T, P.dv)), "dg": np.zeros((st.T, P.dk)),
             "dbeta": np.zeros(st.T), "dh0": np.zeros((P.dk, P.dv))}
        st.so, st.sb = P.dk, 1
        st.dq, st.dk_, st.dv_ = r["dq"].ctypes.data, r["dk"].ctypes.data, r["dv"].ctypes.data
        st.dg, st.dbeta, st.dh0 = r["dg"].ctypes.data, r["dbeta"].ctypes.data, r["dh0"].ctypes.data
        arr[n] = st
        out[(i, h)] = r
    lib().kda_oracle_bwd(arr, len(tasks), n_threads or default_threads())
    return out


def step(q, k, v, beta, g, state, accept_len, *, scale: float = 1.0, eps: float = EPS,
         tasks: Optional[Iterable] = None, n_threads: int = 0):
    """Decode / draft-verify over L tokens per sequence.

    q, k, v, g: [N, L, H, d]; beta: [N, L, H]; state: [N, H, dk, dv]; accept_len: [N].
    Returns ``{(i, h): (o [L, dv], committed state [dk, dv])}``.
    """
    N, L, H, dk = q.shape
    flat = lambda t: t.reshape(N * L, *t.shape[2:])
    cu = torch.arange(0, N * L + 1, L, dtype=torch.int64)
    P = _Prepared(flat(q), flat(k), flat(v), flat(beta), flat(g), cu, state, None, None)
    acc = [int(a) for a in accept_len.to("cpu").tolist()]
    tasks = list(tasks) if tasks is not None else _all_tasks(P)
    arr = (Task * max(1, len(tasks)))()
    out = {}
    for n, (i, h) in enumerate(tasks):
        st = _task(P, i, h, scale, eps)
        st.accept = acc[i]
        o = np.zeros((st.T, P.dv), np.float64)
        hT = np.zeros((P.dk, P.dv), np.float64)
        st.o, st.hT, st.so = o.ctypes.data, hT.ctypes.data, P.dv
        arr[n] = st
        out[(i, h)] = (o, hT)
    lib().kda_oracle_step(arr, len(tasks), n_threads or default_threads())
    return out


def step_paged(q, k, v, beta, g, pool, state_indices, first_slot, accept_len, *, scale: float = 1.0,
               eps: float = EPS, n_threads: int = 0):
    """Two-phase draft/verify over a pool of states (the ReplaySSM rollout pattern of the
    "Kimi K3 on Fireworks" page, rollout section, speculative decoding paragraph).

    Sequence i reads state ``pool[state_indices[i]]``; its token slots before
    ``first_slot[i]`` are padding and are skipped (padding is defined as changing
    nothing), the real tokens run through the token loop of ``step``, and the state is
    committed after ``accept_len[i]`` slots, i.e. after ``accept_len[i] - first_slot[i]``
    real tokens (none if that is not positive).
    Returns ``{(i, h): (o [L - first_slot[i], dv] of the real slots, committed state)}``.
    """
    N, L, H, _ = q.shape
    out = {}
    for i in range(N):
        f, a = int(first_slot[i]), int(accept_len[i])
        sl = slice(i, i + 1)
        slot = int(state_indices[i])
        if f >= L:   # nothing but padding: no outputs, state unchanged
            for h in range(H):
                out[(i, h)] = (np.zeros((0, v.shape[3])), pool[slot, h].double().numpy())
            continue
        r = step(q[sl, f:], k[sl, f:], v[sl, f:], beta[sl, f:], g[sl, f:], pool[slot:slot + 1],
                 torch.tensor([max(0, a - f)], dtype=torch.int32), scale=scale, eps=eps, n_threads=n_threads)
        for h in range(H):
            out[(i, h)] = r[(0, h)]
    return out


def attnres_fwd(sources, w, eps: float = EPS):
    """Attention Residuals forward in fp64 ("Kimi K3 on Fireworks", training section,
    Attention Residuals paragraph; the second page's model figure: alpha = softmax of the
    learned per-sublayer vector against the RMS-normalised sources, then the weighted sum).

    sources: list of S tensors [T, d]; w: [d]. RMSNorm without a gain (any gain folds into w).
    Returns (out [T, d], alpha [T, S], rstd [T, S], logit [T, S]) as float64 numpy arrays.
    """
    X = torch.stack([x.double() for x in sources], 1)              # [T, S, d]
    wd = w.double()
    rstd = (X.pow(2).mean(-1) + eps).rsqrt()                        # [T, S]
    logit = rstd * (X @ wd)                                         # w . (x / rms(x))
    alpha = torch.softmax(logit, -1)
    out = (alpha.unsqueeze(-1) * X).sum(1)
    return out.numpy(), alpha.numpy(), rstd.numpy(), logit.numpy()


def attnres_bwd(sources, w, d_out, eps: float = EPS):
    """Backward of attnres_fwd in fp64, written out step by step (the chain rule through the
    weighted sum, the softmax and the RMS normalisation). Returns (d_sources [S][T, d], dw [d])."""
    X = torch.stack([x.double() for x in sources], 1)              # [T, S, d]
    wd, g = w.double(), d_out.double()
    d = X.shape[-1]
    rstd = (X.pow(2).mean(-1) + eps).rsqrt()
    N = X * rstd.unsqueeze(-1)                                     # normalised sources
    logit = N @ wd
    alpha = torch.softmax(logit, -1)
    # out = sum_i alpha_i x_i
    dX = alpha.unsqueeze(-1) * g.unsqueeze(1)                       # direct path
    dalpha = (X * g.unsqueeze(1)).sum(-1)                           # [T, S]
    dlogit = alpha * (dalpha - (alpha * dalpha).sum(-1, keepdim=True))
    # logit_i = w . n_i:  dn_i = dlogit_i w, dw = sum dlogit_i n_i
    dN = dlogit.unsqueeze(-1) * wd
    dw = (dlogit.unsqueeze(-1) * N).sum((0, 1))
    # n = x r, r = (mean x^2 + eps)^(-1/2):  dx = r (dn - n mean(dn * n))
    dX = dX + rstd.unsqueeze(-1) * (dN - N * (dN * N).sum(-1, keepdim=True) / d)
    return [dX[:, i].numpy() for i in range(X.shape[1])], dw.numpy()


def _conv_bounds(cu_seqlens, n_seqs, total):
    """Per-sequence token ranges: from cu_seqlens, else n_seqs equal sequences."""
    if cu_seqlens is not None:
        cu = [int(c) for c in cu_seqlens.to("cpu").tolist()]
    else:
        n = n_seqs or 1
        cu = [i * (total // n) for i in range(n + 1)]
    return list(zip(cu[:-1], cu[1:]))


def _conv_act(z, activation: str):
    return z / (1.0 + torch.exp(-z)) if activation == "silu" else z


def conv_fwd(x, weight, bias, cu_seqlens, state_in=None, *, activation: str = "silu", n_seqs=None):
    """Short causal depthwise convolution in fp64 (the convolution state named in "Kimi K3 on
    Fireworks: Fast RL at frontier scale", rollout section, inline versus disaggregated
    serving; kernel width, bias and SiLU are this library's reading, stated in include/kda.h).

    Per sequence, the W - 1 state rows (oldest first) are placed before its tokens and every
    output is the tap-weighted sum of the W most recent inputs:
        z[t] = bias + sum_j weight[:, j] * xs[t + j],   xs = [state_in; x_seq]
    x [T, C], weight [C, W], bias [C] or None, state_in [N, W-1, C] or None.
    Returns (y [T, C], state_out [N, W-1, C]) as float64 numpy arrays.
    """
    X, Wt = x.double(), weight.double()
    T, C = X.shape
    W = Wt.shape[1]
    bounds = _conv_bounds(cu_seqlens, n_seqs, T)
    y = torch.zeros(T, C, dtype=torch.float64)
    state_out = torch.zeros(len(bounds), W - 1, C, dtype=torch.float64)
    for n, (s0, s1) in enumerate(bounds):
        prev = state_in[n].double() if state_in is not None else torch.zeros(W - 1, C, dtype=torch.float64)
        xs = torch.cat([prev, X[s0:s1]], 0)
        L = s1 - s0
        z = torch.zeros(L, C, dtype=torch.float64) if bias is None else bias.double().expand(L, C).clone()
        for j in range(W):
            z += Wt[:, j] * xs[j:j + L]
        y[s0:s1] = _conv_act(z, activation)
        state_out[n] = xs[xs.shape[0] - (W - 1):]
    return y.numpy(), state_out.numpy()


def conv_bwd(x, weight, bias, cu_seqlens, state_in, dy, d_state_out=None, *, activation: str = "silu",
             n_seqs=None):
    """Backward of conv_fwd in fp64, by the chain rule written out: dz = dy * act'(z), then every
    tap spreads dz back onto the input row it read (weight[:, j] * dz lands on xs[t + j]) and
    collects dz * xs[t + j] into dweight[:, j]; the gradient of state_out lands on the last W - 1
    rows of xs. Returns dict dx [T, C], dweight [C, W], dbias [C], d_state_in [N, W-1, C] (numpy)."""
    X, Wt, G = x.double(), weight.double(), dy.double()
    T, C = X.shape
    W = Wt.shape[1]
    bounds = _conv_bounds(cu_seqlens, n_seqs, T)
    dx = torch.zeros(T, C, dtype=torch.float64)
    dW = torch.zeros(C, W, dtype=torch.float64)
    db = torch.zeros(C, dtype=torch.float64)
    dst = torch.zeros(len(bounds), W - 1, C, dtype=torch.float64)
    for n, (s0, s1) in enumerate(bounds):
        prev = state_in[n].double() if state_in is not None else torch.zeros(W - 1, C, dtype=torch.float64)
        xs = torch.cat([prev, X[s0:s1]], 0)
        L = s1 - s0
        z = torch.zeros(L, C, dtype=torch.float64) if bias is None else bias.double().expand(L, C).clone()
        for j in range(W):
            z += Wt[:, j] * xs[j:j + L]
        if activation == "silu":
            sg = 1.0 / (1.0 + torch.exp(-z))
            dz = G[s0:s1] * sg * (1.0 + z * (1.0 - sg))
        else:
            dz = G[s0:s1].clone()
        dxs = torch.zeros_like(xs)
        for j in range(W):
            dxs[j:j + L] += Wt[:, j] * dz
            dW[:, j] += (dz * xs[j:j + L]).sum(0)
        db += dz.sum(0)
        if d_state_out is not None and W > 1:
            dxs[xs.shape[0] - (W - 1):] += d_state_out[n].double()
        dx[s0:s1] = dxs[W - 1:]
        dst[n] = dxs[:W - 1]
    return {"dx": dx.numpy(), "dweight": dW.numpy(), "dbias": db.numpy(), "d_state_in": dst.numpy()}


def conv_step(x, weight, bias, pool, state_indices=None, accept_len=None, first_slot=None, *,
              activation: str = "silu"):
    """Decode / verify form of conv_fwd in fp64: x [N, L, C] token slots per sequence, pool
    [P, W-1, C] states. Slots before first_slot[i] are padding (no output, no state change);
    sequence i convolves slots first_slot[i]..L-1 from the state of its slot and commits the
    last W - 1 inputs of slots up to accept_len[i] (nothing when accept_len[i] <= first_slot[i]).
    Returns (y [N, L, C] with NaN in padding slots, new pool) as float64 numpy arrays."""
    X, Wt = x.double(), weight.double()
    N, L, C = X.shape
    W = Wt.shape[1]
    new_pool = pool.double().clone()
    y = torch.full((N, L, C), float("nan"), dtype=torch.float64)
    for n in range(N):
        slot = int(state_indices[n]) if state_indices is not None else n
        F = min(max(int(first_slot[n]), 0), L) if first_slot is not None else 0
        a = min(max(int(accept_len[n]), 0), L) if accept_len is not None else L
        xs = torch.cat([pool[slot].double(), X[n, F:]], 0)
        Lt = L - F
        z = torch.zeros(Lt, C, dtype=torch.float64) if bias is None else bias.double().expand(Lt, C).clone()
        for j in range(W):
            z += Wt[:, j] * xs[j:j + Lt]
        y[n, F:] = _conv_act(z, activation)
        if a > F:
            kept = xs[:W - 1 + a - F]
            new_pool[slot] = kept[kept.shape[0] - (W - 1):]
    return y.numpy(), new_pool.numpy()


def assemble_fwd(res: dict, cu_seqlens, H: int, dv: int):
    """Stack per-task forward results into o [total, H, dv] and hT [N, H, dk, dv]."""
    cu = [int(x) for x in cu_seqlens.to("cpu").tolist()]
    N = len(cu) - 1
    dk = next(iter(res.values()))[1].shape[0]
    o = np.zeros((cu[-1], H, dv))
    hT = np.zeros((N, H, dk, dv))
    for (i, h), (oi, hi) in res.items():
        o[cu[i]:cu[i + 1], h] = oi
        hT[i, h] = hi
    return o, hT


def assemble_bwd(res: dict, cu_seqlens, H: int):
    cu = [int(x) for x in cu_seqlens.to("cpu").tolist()]
    N = len(cu) - 1
    any_r = next(iter(res.values()))
    dk, dv = any_r["dq"].shape[1], any_r["dv"].shape[1]
    out = {"dq": np.zeros((cu[-1], H, dk)), "dk": np.zeros((cu[-1], H, dk)),
           "dv": np.zeros((cu[-1], H, dv)), "dg": np.zeros((cu[-1], H, dk)),
           "dbeta": np.zeros((cu[-1], H)), "dh0": np.zeros((N, H, dk, dv))}
    for (i, h), r in res.items():
        for name in ("dq", "dk", "dv", "dg", "dbeta"):
            out[name][cu[i]:cu[i + 1], h] = r[name]
        out["dh0"][i, h] = r["dh0"]
    return out
