"""GB300-native Kimi Delta Attention (KDA): chunked forward, backward and decode.

Python face of libkda.so (include/kda.h). Every step of the computation runs in
the library's CUDA kernels; this module only allocates outputs and workspaces
with PyTorch, passes raw device pointers and the current CUDA stream through
ctypes, and turns status codes into exceptions.

    o, hT, saved = kda_fwd(q, k, v, beta, g, cu_seqlens, h0, save=True)
    grads = kda_bwd(q, k, v, beta, g, dO, saved, cu_seqlens, h0, dhT)
    o = kda_step(q, k, v, beta, g, state, accept_len)     # state updated in place

Shapes: q, k, v, g, dO [total, H, 128]; beta [total, H]; states [N, H, 128, 128]
(fp32, [key][value]); decode inputs carry an extra step axis: [N, L, H, ...].
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _lib
from ._lib import KdaError

__all__ = ["kda_fwd", "kda_bwd", "kda_step", "fwd_args", "bwd_args", "KdaError", "library"]


def library():
    """The loaded libkda.so handle (raises if it was not built)."""
    return _lib.load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.KDA_BF16
    if t.dtype == torch.float32:
        return _lib.KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_inputs(q, k, v, beta, g):
    for name, t in (("q", q), ("k", k), ("v", v), ("beta", beta), ("g", g)):
        if t is None and name == "v":
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if beta.dtype != torch.float32 or g.dtype != torch.float32:
        raise TypeError("beta and g must be float32")
    if k.dtype != q.dtype or (v is not None and v.dtype != q.dtype):
        raise TypeError("q, k and v must share one dtype")


def fwd_args(q, k, v, beta, g, cu_seqlens=None, h0=None, o=None, hT=None, saved=None,
             workspace=None, scale: float = 1.0, n_seqs: Optional[int] = None, dev_status=None,
             h0_identity: bool = False) -> _lib.FwdArgs:
    """Fill the C argument struct for kda_fwd from tensors (no allocation)."""
    a = _lib.FwdArgs()
    total, H, dk = q.shape
    a.n_seqs = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (n_seqs or 1)
    a.total_tokens, a.heads, a.dk, a.dv, a.chunk = total, H, dk, (v.shape[2] if v is not None else dk), 64
    a.h0_identity = int(h0_identity)
    a.scale, a.io_dtype = scale, _io_dtype(q)
    a.cu_seqlens = _ptr(cu_seqlens)
    a.q, a.k, a.v, a.beta, a.g = _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g)
    a.h0, a.o, a.hT, a.saved = _ptr(h0), _ptr(o), _ptr(hT), _ptr(saved)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    a.dev_status = _ptr(dev_status)
    return a


def bwd_args(fa: _lib.FwdArgs, dO, dq, dk, dv, dbeta, dg, dh0=None, dhT=None, workspace=None) -> _lib.BwdArgs:
    b = _lib.BwdArgs()
    b.fwd = fa
    b.dO, b.dhT = _ptr(dO), _ptr(dhT)
    b.dq, b.dk, b.dv, b.dbeta, b.dg, b.dh0 = _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(dh0)
    b.workspace = _ptr(workspace)
    b.workspace_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return b


def _i32(cu_seqlens, device):
    if cu_seqlens is None:
        return None
    if cu_seqlens.device.type == "cpu":
        # through pinned memory, so the copy is enqueued on the current stream instead of
        # blocking the host until the stream reaches it
        return cu_seqlens.to(dtype=torch.int32).contiguous().pin_memory().to(device, non_blocking=True)
    return cu_seqlens.to(device=device, dtype=torch.int32).contiguous()


def kda_fwd(q, k, v, beta, g, cu_seqlens=None, h0=None, *, scale: float = 1.0, save: bool = False,
            final_state: bool = True, n_seqs: Optional[int] = None, dev_status=None):
    """Chunked KDA forward. Returns (o, hT or None, saved or None).

    ``saved`` (chunk-start states) is what kda_bwd needs; request it with save=True.
    Without cu_seqlens the tokens form ``n_seqs`` (default 1) equal sequences.
    ``dev_status`` (optional int32 device tensor, zeroed by the caller) receives
    KDA_ERR_TIMEOUT if a kernel gives up a bounded wait.
    """
    lib = library()
    _check_inputs(q, k, v, beta, g)
    dev = q.device
    cu = _i32(cu_seqlens, dev)
    N = (cu.numel() - 1) if cu is not None else (n_seqs or 1)
    H = q.shape[1]
    o = torch.empty_like(v)
    hT = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev) if final_state else None
    a = fwd_args(q, k, v, beta, g, cu, h0, o, hT, None, None, scale, n_seqs=N, dev_status=dev_status)
    saved = None
    if save:
        saved = torch.empty(lib.kda_saved_size(C.byref(a)), dtype=torch.uint8, device=dev)
        a.saved = saved.data_ptr()
    ws_bytes = lib.kda_fwd_workspace_size(C.byref(a))
    if ws_bytes == 0:
        _lib.check(lib.kda_fwd(C.byref(a), _stream(dev)))   # reports the argument error
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_fwd(C.byref(a), _stream(dev)))
    return o, hT, saved


def _fwd_states(q, k, v, beta, g, cu, h0, N, *, scale, h0_identity=False, out=None, ws=None):
    """One forward pass for its final states (and outputs into ``out`` when given). With
    ``ws`` (the workspace of an earlier pass on the same q, k, g, beta, cu) the chunk records
    are reused and only the scan runs; returns (hT, workspace)."""
    lib = library()
    dev = q.device
    hT = torch.empty((N, q.shape[1], 128, 128), dtype=torch.float32, device=dev)
    a = fwd_args(q, k, v, beta, g, cu, h0, out, hT, None, None, scale, n_seqs=N, h0_identity=h0_identity)
    ws_bytes = lib.kda_fwd_workspace_size(C.byref(a))
    if ws is None:
        ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    else:
        a.skip_prep = 1
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_fwd(C.byref(a), _stream(dev)))
    return hT, ws


def kda_cp_combine(M, b, h0, n_segments: int):
    """States entering each segment: S_in[:, 0] = h0, S_in[:, k+1] = M[:, k] S_in[:, k] + b[:, k].

    M, b: [N, P, H, 128, 128] fp32 (maps and offsets of the segments); h0: [N, H, 128, 128]
    fp32 or None. Returns S_in [N, P, H, 128, 128].
    """
    lib = library()
    N, P, H = M.shape[:3]
    if P != n_segments or b.shape != M.shape or (h0 is not None and h0.shape != (N, H, 128, 128)):
        raise ValueError("M, b must be [N, P, H, 128, 128] and h0 [N, H, 128, 128]")
    s_in = torch.empty_like(M)
    a = _lib.CpArgs(N, P, H, 128, 128, M.data_ptr(), b.data_ptr(), _ptr(h0), s_in.data_ptr())
    _lib.check(lib.kda_cp_combine(C.byref(a), _stream(M.device)))
    return s_in


def kda_fwd_cp(q, k, v, beta, g, cu_seqlens=None, h0=None, *, n_segments: int, scale: float = 1.0,
               n_seqs: Optional[int] = None, dev_status=None):
    """Forward by context parallelism, emulated on one device (libkda's kda_fwd_cp): every
    sequence is cut into n_segments consecutive runs of whole chunks that are processed
    independently (as separate sequences), their affine maps combined, and the segments run
    again from the combined incoming states. Returns (o, hT) of the unsplit forward.
    """
    lib = library()
    _check_inputs(q, k, v, beta, g)
    dev = q.device
    cu = _i32(cu_seqlens, dev)
    N = (cu.numel() - 1) if cu is not None else (n_seqs or 1)
    H = q.shape[1]
    o = torch.empty_like(v)
    hT = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
    c = _lib.FwdCpArgs()
    c.fwd = fwd_args(q, k, v, beta, g, cu, None if h0 is None else h0.contiguous(), o, hT, None, None, scale,
                     n_seqs=N, dev_status=dev_status)
    c.n_segments = n_segments
    ws_bytes = lib.kda_fwd_cp_workspace_size(C.byref(c))
    if ws_bytes == 0:
        raise KdaError(_lib.KDA_ERR_INVALID_ARG, lib.kda_last_error().decode())
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    c.workspace, c.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_fwd_cp(C.byref(c), _stream(dev)))
    return o, hT


def _attnres_args(sources, w, eps, out=None, stats=None):
    S = len(sources)
    if not 1 <= S <= _lib.ATTNRES_MAX_SOURCES:
        raise ValueError("Attention Residuals takes 1..9 sources")
    T, d = sources[0].shape
    for x in sources:
        if x.shape != (T, d) or x.dtype != sources[0].dtype or not x.is_cuda or not x.is_contiguous():
            raise ValueError("sources must be contiguous CUDA tensors of one shape [T, d] and dtype")
    if w.dtype != torch.float32 or w.shape != (d,) or not w.is_contiguous():
        raise TypeError("w must be a contiguous float32 [d] tensor")
    a = _lib.AttnresFwdArgs()
    a.n_sources, a.tokens, a.dim, a.eps, a.io_dtype = S, T, d, eps, _io_dtype(sources[0])
    for i, x in enumerate(sources):
        a.src[i] = x.data_ptr()
    a.w, a.out = w.data_ptr(), _ptr(out)
    a.alpha, a.rstd, a.logit = (_ptr(t) for t in stats)
    return a


def attnres_fwd(sources, w, *, eps: float = 1e-6):
    """Attention Residuals forward: out = sum_i softmax_i(r_i (w . x_i)) x_i over the sources
    (r_i = 1 / RMS(x_i)). Returns (out [T, d], stats) with stats = (alpha, rstd, logit), each
    [T, S] fp32, which the backward takes."""
    lib = library()
    T, d = sources[0].shape
    dev = sources[0].device
    out = torch.empty_like(sources[0])
    stats = tuple(torch.empty((T, len(sources)), dtype=torch.float32, device=dev) for _ in range(3))
    a = _attnres_args(sources, w, eps, out, stats)
    _lib.check(lib.kda_attnres_fwd(C.byref(a), _stream(dev)))
    return out, stats


def attnres_bwd(sources, w, stats, d_out, *, eps: float = 1e-6):
    """Backward of attnres_fwd: returns (d_sources list, dw [d] fp32)."""
    lib = library()
    dev = sources[0].device
    if d_out.shape != sources[0].shape or d_out.dtype != sources[0].dtype or not d_out.is_contiguous():
        raise ValueError("d_out must match the sources")
    b = _lib.AttnresBwdArgs()
    b.fwd = _attnres_args(sources, w, eps, None, stats)
    d_src = [torch.empty_like(x) for x in sources]
    dw = torch.empty_like(w)
    b.d_out, b.dw = d_out.data_ptr(), dw.data_ptr()
    for i, x in enumerate(d_src):
        b.d_src[i] = x.data_ptr()
    ws_bytes = lib.kda_attnres_bwd_workspace_size(C.byref(b))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    b.workspace, b.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_attnres_bwd(C.byref(b), _stream(dev)))
    return d_src, dw


_ACT = {"none": _lib.KDA_ACT_NONE, "silu": _lib.KDA_ACT_SILU}


def _conv_args(x, weight, bias, cu, state_in, activation, n_seqs):
    if x.dim() != 2 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [T, C]")
    T, Cc = x.shape
    if weight.dtype != torch.float32 or weight.dim() != 2 or weight.shape[0] != Cc or not weight.is_contiguous():
        raise TypeError("weight must be a contiguous float32 [C, W] tensor")
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (Cc,)):
        raise TypeError("bias must be float32 [C]")
    W = weight.shape[1]
    if state_in is not None and (state_in.dtype != x.dtype or state_in.shape != (n_seqs, W - 1, Cc)
                                 or not state_in.is_contiguous()):
        raise ValueError("state_in must be a contiguous [N, W-1, C] tensor of x's dtype")
    a = _lib.ConvArgs()
    a.n_seqs, a.total_tokens, a.channels, a.width = n_seqs, T, Cc, W
    a.activation, a.io_dtype = _ACT[activation], _io_dtype(x)
    a.cu_seqlens, a.x, a.weight, a.bias, a.state_in = _ptr(cu), x.data_ptr(), weight.data_ptr(), _ptr(bias), _ptr(state_in)
    return a


def conv_fwd(x, weight, bias=None, cu_seqlens=None, state_in=None, *, activation: str = "silu",
             n_seqs: Optional[int] = None):
    """Short causal depthwise convolution (width W = weight.shape[1]) with the convolution
    state of each sequence. Returns (y [T, C] in x's dtype, state_out [N, W-1, C])."""
    lib = library()
    cu = _i32(cu_seqlens, x.device)
    N = (cu.numel() - 1) if cu is not None else (n_seqs or 1)
    a = _conv_args(x, weight, bias, cu, state_in, activation, N)
    y = torch.empty_like(x)
    state_out = torch.empty((N, weight.shape[1] - 1, x.shape[1]), dtype=x.dtype, device=x.device)
    a.y, a.state_out = y.data_ptr(), _ptr(state_out) if state_out.numel() else None
    _lib.check(lib.kda_conv_fwd(C.byref(a), _stream(x.device)))
    return y, state_out


def conv_bwd(x, weight, bias, dy, cu_seqlens=None, state_in=None, d_state_out=None, *, activation: str = "silu",
             n_seqs: Optional[int] = None):
    """Backward of conv_fwd: returns a dict of fp32 gradients dx, dweight, dbias (None without a
    bias) and d_state_in."""
    lib = library()
    cu = _i32(cu_seqlens, x.device)
    N = (cu.numel() - 1) if cu is not None else (n_seqs or 1)
    if dy.shape != x.shape or dy.dtype != x.dtype or not dy.is_contiguous():
        raise ValueError("dy must match x")
    b = _lib.ConvBwdArgs()
    b.fwd = _conv_args(x, weight, bias, cu, state_in, activation, N)
    f32 = dict(dtype=torch.float32, device=x.device)
    W = weight.shape[1]
    dx, dweight = torch.empty(x.shape, **f32), torch.empty(weight.shape, **f32)
    dbias = torch.empty(x.shape[1], **f32) if bias is not None else None
    d_state_in = torch.empty((N, W - 1, x.shape[1]), **f32)
    if d_state_out is not None:
        d_state_out = d_state_out.to(torch.float32).contiguous()
    b.dy, b.d_state_out, b.dx, b.dweight = dy.data_ptr(), _ptr(d_state_out), dx.data_ptr(), dweight.data_ptr()
    b.dbias, b.d_state_in = _ptr(dbias), _ptr(d_state_in) if d_state_in.numel() else None
    ws_bytes = lib.kda_conv_bwd_workspace_size(C.byref(b))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=x.device)
    b.workspace, b.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_conv_bwd(C.byref(b), _stream(x.device)))
    return {"dx": dx, "dweight": dweight, "dbias": dbias, "d_state_in": d_state_in}


def conv_step(x, weight, bias, state, accept_len=None, *, activation: str = "silu", state_indices=None,
              first_slot=None, out=None, dev_status=None):
    """Decode / verify L token slots per sequence through the short convolution: x [N, L, C];
    ``state`` [N, W-1, C] (or a pool [P, W-1, C] addressed by ``state_indices``) advanced in
    place through ``accept_len`` slots; slots before ``first_slot`` are padding. Returns y."""
    lib = library()
    if x.dim() != 3 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor [N, L, C]")
    N, L, Cc = x.shape
    W = weight.shape[1]
    if state.dtype != x.dtype or state.shape[1:] != (W - 1, Cc) or not state.is_contiguous():
        raise ValueError("state must be a contiguous [P, W-1, C] tensor of x's dtype")
    i32 = lambda t: None if t is None else t.to(device=x.device, dtype=torch.int32).contiguous()
    acc, idx, first = i32(accept_len), i32(state_indices), i32(first_slot)
    if (idx is None and state.shape[0] != N) or (idx is not None and idx.numel() != N):
        raise ValueError("state has one slot per sequence unless state_indices [N] addresses a pool")
    y = torch.empty_like(x) if out is None else out
    a = _lib.ConvStepArgs()
    a.n_seqs, a.steps, a.channels, a.width = N, L, Cc, W
    a.activation, a.io_dtype = _ACT[activation], _io_dtype(x)
    a.x, a.weight, a.bias, a.state = x.data_ptr(), weight.data_ptr(), _ptr(bias), _ptr(state) if state.numel() else None
    a.state_indices, a.n_slots, a.accept_len, a.first_slot = _ptr(idx), state.shape[0], _ptr(acc), _ptr(first)
    a.y, a.dev_status = y.data_ptr(), _ptr(dev_status)
    _lib.check(lib.kda_conv_step(C.byref(a), _stream(x.device)))
    return y


def kda_bwd(q, k, v, beta, g, dO, saved, cu_seqlens=None, h0=None, dhT=None, *, scale: float = 1.0,
            n_seqs: Optional[int] = None, initial_state_grad: bool = True, dev_status=None, out=None):
    """Backward of kda_fwd (``saved`` from kda_fwd(..., save=True) with the same inputs).

    Returns a dict of fp32 gradients: dq, dk, dv, dbeta, dg and dh0 (or None). ``out``, a dict
    with the same keys, supplies the gradient tensors to write (contiguous fp32 of the inputs'
    shapes; dh0 [N, H, 128, 128]) instead of fresh ones.
    """
    lib = library()
    _check_inputs(q, k, v, beta, g)
    dev = q.device
    cu = _i32(cu_seqlens, dev)
    N = (cu.numel() - 1) if cu is not None else (n_seqs or 1)
    H = q.shape[1]
    f32 = dict(dtype=torch.float32, device=dev)
    if out is not None:
        want = {"dq": q.shape, "dk": k.shape, "dv": v.shape, "dg": g.shape, "dbeta": beta.shape}
        for name, shape in want.items():
            t = out[name]
            if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != dev:
                raise ValueError(f"out[{name!r}] must be a contiguous float32 tensor of shape {tuple(shape)} on {dev}")
        dq, dk, dv, dg, dbeta = (out[n] for n in ("dq", "dk", "dv", "dg", "dbeta"))
        dh0 = out.get("dh0") if initial_state_grad else None
        if dh0 is not None and (dh0.dtype != torch.float32 or tuple(dh0.shape) != (N, H, 128, 128)
                                or not dh0.is_contiguous()):
            raise ValueError("out['dh0'] must be a contiguous float32 [N, H, 128, 128] tensor")
    else:
        dq, dk, dv = torch.empty(q.shape, **f32), torch.empty(k.shape, **f32), torch.empty(v.shape, **f32)
        dg, dbeta = torch.empty(g.shape, **f32), torch.empty(beta.shape, **f32)
        dh0 = torch.empty((N, H, 128, 128), **f32) if initial_state_grad else None
    fa = fwd_args(q, k, v, beta, g, cu, h0, None, None, saved, None, scale, n_seqs=N, dev_status=dev_status)
    b = bwd_args(fa, dO, dq, dk, dv, dbeta, dg, dh0, dhT)
    ws_bytes = lib.kda_bwd_workspace_size(C.byref(b))
    if ws_bytes == 0:
        _lib.check(lib.kda_bwd(C.byref(b), _stream(dev)))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    b.workspace, b.workspace_bytes = ws.data_ptr(), ws_bytes
    _lib.check(lib.kda_bwd(C.byref(b), _stream(dev)))
    return {"dq": dq, "dk": dk, "dv": dv, "dbeta": dbeta, "dg": dg, "dh0": dh0}


def step_args(q, k, v, beta, g, state, accept_len, o, scale: float = 1.0, state_indices=None,
              first_slot=None, dev_status=None) -> _lib.StepArgs:
    a = _lib.StepArgs()
    N, L, H, dk = q.shape
    a.n_seqs, a.steps, a.heads, a.dk, a.dv = N, L, H, dk, v.shape[3]
    a.scale, a.io_dtype = scale, _io_dtype(q)
    a.q, a.k, a.v, a.beta, a.g = _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g)
    a.state, a.accept_len, a.o = _ptr(state), _ptr(accept_len), _ptr(o)
    a.state_indices, a.first_slot, a.dev_status = _ptr(state_indices), _ptr(first_slot), _ptr(dev_status)
    a.n_slots = state.shape[0]
    return a


def kda_step(q, k, v, beta, g, state, accept_len=None, *, scale: float = 1.0, out=None, state_indices=None,
             first_slot=None, dev_status=None):
    """Decode / draft-verify L tokens per sequence; returns o [N, L, H, 128].

    ``state`` [N, H, 128, 128] fp32 (or a pool [P, H, 128, 128] addressed by
    ``state_indices`` [N]) is overwritten with the state after ``accept_len[i]`` token
    slots (left untouched where accept_len is 0; all L when None). Slots before
    ``first_slot[i]`` are padding: no state change, output not written. See
    include/kda.h for the verify-then-replay use of the two.
    """
    lib = library()
    _check_inputs(q, k, v, beta, g)
    if state.dtype != torch.float32 or not state.is_contiguous():
        raise TypeError("state must be a contiguous float32 tensor")
    i32 = lambda t: None if t is None else t.to(device=q.device, dtype=torch.int32).contiguous()
    acc, idx, first = i32(accept_len), i32(state_indices), i32(first_slot)
    N = q.shape[0]
    if (idx is None and state.shape[0] != N) or (idx is not None and idx.numel() != N):
        raise ValueError("state has one slot per sequence unless state_indices [N] addresses a pool")
    if first is not None and first.numel() != N:
        raise ValueError("first_slot must have one entry per sequence")
    o = torch.empty_like(v) if out is None else out
    a = step_args(q, k, v, beta, g, state, acc, o, scale, idx, first, dev_status)
    _lib.check(lib.kda_step(C.byref(a), _stream(q.device)))
    return o
