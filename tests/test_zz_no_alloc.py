"""kda_fwd_no_alloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an engine that owns all device memory, or a path
that cannot take cudaMalloc's device synchronisation) pass only inputs and
outputs; the scratch comes from a fixed static device array. The entry point is
checked here through the C ABI against kda_fwd (with a caller-allocated
workspace) on two calls in a row, and it must reject problems whose scratch
would exceed the static array. This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gated_delta_rule_chunked_gb300.inputs import make_seq_batch

pytestmark = pytest.mark.gpu

TOL = 1e-2   # max|diff| / max|ref|, the bf16 parity tolerance of the other tests


def rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def test_no_alloc_forward_matches_kda_fwd_twice():
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    lib = kda.library()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call, seed in enumerate((21, 22)):
        b = make_seq_batch([300, 77, 129], heads=4, io_dtype="bf16", seed=seed, h0=True)
        t = {n: getattr(b, n).to(dev) for n in ("q", "k", "v", "beta", "g", "cu_seqlens", "h0")}
        N, H = 3, 4
        # reference: the existing entry point with a caller-allocated workspace
        o_ref = torch.empty_like(t["v"])
        h_ref = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
        a = kda.fwd_args(t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"], o_ref, h_ref)
        ws = torch.empty(lib.kda_fwd_workspace_size(C.byref(a)), dtype=torch.uint8, device=dev)
        a = kda.fwd_args(t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"], o_ref, h_ref, None, ws)
        _lib.check(lib.kda_fwd(C.byref(a), stream))
        # the no-allocation entry point: no workspace passed
        o = torch.full_like(t["v"], float("nan"))
        hT = torch.full((N, H, 128, 128), float("nan"), dtype=torch.float32, device=dev)
        a2 = kda.fwd_args(t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"], o, hT)
        assert a2.workspace is None and a2.workspace_bytes == 0
        _lib.check(lib.kda_fwd_no_alloc(C.byref(a2), stream))
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(hT).all(), f"call {call}"
        assert rel(o.float(), o_ref.float()) <= TOL, f"call {call}"
        assert rel(hT, h_ref) <= TOL, f"call {call}"


def test_no_alloc_rejects_problems_beyond_the_static_scratch():
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    lib = kda.library()
    a = _lib.FwdArgs()
    a.n_seqs, a.total_tokens, a.heads, a.dk, a.dv, a.chunk = 1, 1 << 20, 96, 128, 128, 64
    a.scale, a.io_dtype = 1.0, _lib.KDA_BF16
    fake = 1 << 40      # never dereferenced: the size check comes first
    a.q = a.k = a.v = a.g = a.o = a.beta = fake
    assert lib.kda_fwd_workspace_size(C.byref(a)) > _lib.NO_ALLOC_SCRATCH_BYTES
    assert lib.kda_fwd_no_alloc(C.byref(a), None) == _lib.KDA_ERR_INVALID_ARG
    assert "static scratch" in lib.kda_last_error().decode()
