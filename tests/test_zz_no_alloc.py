"""kda_fwd_no_alloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an engine that owns all device memory, or a path
that cannot take cudaMalloc's device synchronisation) pass only inputs and
outputs; the scratch comes from a fixed static device array. The entry point is
checked here through the C ABI against kda_fwd (with a caller-allocated
workspace) on two calls in a row. Both run the same deterministic kernels on the
same inputs, so their outputs must be bit-identical: a stale or misplaced scratch
read would show up as a difference. It must also ignore the caller's workspace
fields, reject skip_prep (the shared scratch may hold another call's records) and
reject problems whose scratch would exceed the static array. This file is
collected last on purpose.
"""
import ctypes as C

import pytest
import torch

from gated_delta_rule_chunked_gb300.inputs import make_seq_batch

pytestmark = pytest.mark.gpu


def _case(dev, lens, heads, io_dtype, seed):
    b = make_seq_batch(lens, heads=heads, io_dtype=io_dtype, seed=seed, h0=True)
    t = {n: getattr(b, n).to(dev) for n in ("q", "k", "v", "beta", "g", "cu_seqlens", "h0")}
    N, H = len(lens), heads
    args = (t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"])
    return t, N, H, args


@pytest.mark.parametrize("io_dtype,save", [("bf16", False), ("f32", False), ("bf16", True)])
def test_no_alloc_forward_bit_identical_to_kda_fwd_twice(io_dtype, save):
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    lib = kda.library()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call, seed in enumerate((21, 22)):
        t, N, H, args = _case(dev, [300, 77, 129], 4, io_dtype, seed + (10 if save else 0))
        # reference: the existing entry point with a caller-allocated workspace
        o_ref = torch.empty_like(t["v"])
        h_ref = torch.empty((N, H, 128, 128), dtype=torch.float32, device=dev)
        a = kda.fwd_args(*args, o_ref, h_ref)
        # both saved buffers start from the same fill: slots past the real chunks are not written
        sv_ref = torch.full((lib.kda_saved_size(C.byref(a)),), 0xA5, dtype=torch.uint8, device=dev) if save else None
        a = kda.fwd_args(*args, o_ref, h_ref, sv_ref)
        ws = torch.empty(lib.kda_fwd_workspace_size(C.byref(a)), dtype=torch.uint8, device=dev)
        a = kda.fwd_args(*args, o_ref, h_ref, sv_ref, ws)
        _lib.check(lib.kda_fwd(C.byref(a), stream))
        # the no-allocation entry point: no workspace, or a stale one that it must ignore
        o = torch.full_like(t["v"], float("nan"))
        hT = torch.full((N, H, 128, 128), float("nan"), dtype=torch.float32, device=dev)
        sv = torch.full_like(sv_ref, 0xA5) if save else None
        a2 = kda.fwd_args(*args, o, hT, sv)
        if call == 1:
            a2.workspace, a2.workspace_bytes = 3, 5      # misaligned and too small: ignored
        else:
            assert a2.workspace is None and a2.workspace_bytes == 0
        _lib.check(lib.kda_fwd_no_alloc(C.byref(a2), stream))
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), f"call {call}: o differs from kda_fwd"
        assert torch.equal(hT, h_ref), f"call {call}: hT differs from kda_fwd"
        if save:
            assert torch.equal(sv, sv_ref), f"call {call}: saved differs from kda_fwd"


def test_no_alloc_rejects_skip_prep():
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    lib = kda.library()
    dev = torch.device("cuda")
    t, N, H, args = _case(dev, [128], 2, "bf16", 23)
    o = torch.full_like(t["v"], 7.0)
    a = kda.fwd_args(*args, o, None)
    a.skip_prep = 1
    assert lib.kda_fwd_no_alloc(C.byref(a), None) == _lib.KDA_ERR_UNSUPPORTED
    assert "skip_prep" in lib.kda_last_error().decode()
    torch.cuda.synchronize()
    assert torch.all(o.float() == 7.0)                 # nothing was enqueued


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
