"""A bounded wait that runs out, on the GPU, without a fault or a hang.

Every mbarrier wait of the kernels gives up after a time limit, writes
KDA_ERR_TIMEOUT to the caller's status word and lets the CTA leave. Here the
forward scan's first CTA (sequence 0, head 0) is told not to issue its first
copies (kda_fwd_args.debug_starve), so nothing of it is in flight and its waits
can only run out; the limit is set to 1 ms (wait_limit_ns). The test checks the
status word, that the starved head's outputs were left alone while the other
head's match the oracle, and that the context still runs a normal call.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_chunked_gb300.inputs import make_seq_batch

pytestmark = pytest.mark.gpu


def rel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))


def test_starved_scan_wait_runs_out_and_reports_timeout():
    import gated_delta_rule_chunked_gb300 as kda
    from gated_delta_rule_chunked_gb300 import _lib
    lib = kda.library()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev).cuda_stream
    b = make_seq_batch([200], heads=2, io_dtype="bf16", seed=81, h0=True)
    t = {n: getattr(b, n).to(dev) for n in ("q", "k", "v", "beta", "g", "cu_seqlens", "h0")}
    args = (t["q"], t["k"], t["v"], t["beta"], t["g"], t["cu_seqlens"], t["h0"])
    ref = oracle.fwd(b.q, b.k, b.v, b.beta, b.g, b.cu_seqlens, b.h0)
    o_ref, h_ref = oracle.assemble_fwd(ref, b.cu_seqlens, 2, 128)

    def run(starve):
        o = torch.full_like(t["v"], 7.0)
        hT = torch.full((1, 2, 128, 128), 7.0, dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        a = kda.fwd_args(*args, o, hT)
        ws = torch.empty(lib.kda_fwd_workspace_size(C.byref(a)), dtype=torch.uint8, device=dev)
        a = kda.fwd_args(*args, o, hT, None, ws, dev_status=status)
        a.wait_limit_ns = 1_000_000          # 1 ms
        a.debug_starve = int(starve)
        _lib.check(lib.kda_fwd(C.byref(a), stream))
        torch.cuda.synchronize()
        return o, hT, int(status.item())

    o, hT, st = run(True)
    assert st == _lib.KDA_ERR_TIMEOUT
    assert torch.all(o[:, 0].float() == 7.0) and torch.all(hT[0, 0] == 7.0)   # the starved head: untouched
    assert rel(o[:, 1].float().cpu(), o_ref[:, 1]) <= 1e-2                    # the other head: computed
    assert rel(hT[0, 1].cpu(), h_ref[0, 1]) <= 1e-2
    # the context is still usable: a normal call with the same short limit completes and matches
    o, hT, st = run(False)
    assert st == 0
    assert rel(o.float().cpu(), o_ref) <= 1e-2 and rel(hT.cpu(), h_ref) <= 1e-2
