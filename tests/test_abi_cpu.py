"""CPU checks of the C ABI: the library loads, exports every declared symbol,
the ctypes structs match the C layout, and argument validation rejects bad
calls before anything touches a GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_chunked_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    from gated_delta_rule_chunked_gb300 import _lib
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", os.path.join(ROOT, "gated_delta_rule_chunked_gb300",
                                                                     "libkda.so")],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kda_\w+)", out))
    assert set(declared_functions()) <= exported


def test_abi_version(lib):
    assert lib.kda_abi_version() == 5


def test_struct_layout_matches_c(tmp_path):
    from gated_delta_rule_chunked_gb300 import _lib
    probe = tmp_path / "probe.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kda.h"', "int main(void){"]
    for sname, cls in (("kda_fwd_args", _lib.FwdArgs), ("kda_bwd_args", _lib.BwdArgs),
                       ("kda_step_args", _lib.StepArgs), ("kda_cp_args", _lib.CpArgs),
                       ("kda_fwd_cp_args", _lib.FwdCpArgs),
                       ("kda_attnres_fwd_args", _lib.AttnresFwdArgs), ("kda_attnres_bwd_args", _lib.AttnresBwdArgs),
                       ("kda_conv_args", _lib.ConvArgs), ("kda_conv_bwd_args", _lib.ConvBwdArgs),
                       ("kda_conv_step_args", _lib.ConvStepArgs)):
        lines.append(f'printf("{sname} %zu\\n", sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{sname}.{fname} %zu\\n", offsetof({sname}, {fname}));')
    lines.append("return 0;}")
    probe.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                           str(probe), "-o", str(exe)])
    got = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    for sname, cls in (("kda_fwd_args", _lib.FwdArgs), ("kda_bwd_args", _lib.BwdArgs),
                       ("kda_step_args", _lib.StepArgs), ("kda_cp_args", _lib.CpArgs),
                       ("kda_fwd_cp_args", _lib.FwdCpArgs),
                       ("kda_attnres_fwd_args", _lib.AttnresFwdArgs), ("kda_attnres_bwd_args", _lib.AttnresBwdArgs),
                       ("kda_conv_args", _lib.ConvArgs), ("kda_conv_bwd_args", _lib.ConvBwdArgs),
                       ("kda_conv_step_args", _lib.ConvStepArgs)):
        assert int(got[sname]) == C.sizeof(cls), sname
        for fname, _ in cls._fields_:
            assert int(got[f"{sname}.{fname}"]) == getattr(cls, fname).offset, f"{sname}.{fname}"


def _fwd_args(**over):
    from gated_delta_rule_chunked_gb300 import _lib
    a = _lib.FwdArgs()
    a.n_seqs, a.total_tokens, a.heads, a.dk, a.dv, a.chunk = 1, 128, 2, 128, 128, 64
    a.scale, a.io_dtype = 1.0, _lib.KDA_BF16
    fake = 1 << 40          # well-aligned, never dereferenced: validation fails first
    a.q = a.k = a.v = a.g = a.o = a.beta = fake
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("field,value,status", [
    ("dk", 64, 2), ("chunk", 32, 2), ("io_dtype", 7, 2),
    ("heads", 0, 1), ("n_seqs", 0, 1), ("total_tokens", -1, 1),
    ("q", None, 1), ("g", (1 << 40) + 8, 1), ("total_tokens", 127, 1),   # 127 not divisible? n_seqs=1 ok
])
def test_fwd_validation_rejects_before_launch(lib, field, value, status):
    from gated_delta_rule_chunked_gb300 import _lib
    if field == "total_tokens" and value == 127:
        a = _fwd_args(n_seqs=2, total_tokens=127)      # equal-length split impossible
    else:
        a = _fwd_args(**{field: value})
    assert lib.kda_fwd(C.byref(a), None) == status
    assert lib.kda_last_error().decode()


def test_fwd_rejects_small_workspace(lib):
    a = _fwd_args()
    need = lib.kda_fwd_workspace_size(C.byref(a))
    assert need > 0
    a.workspace, a.workspace_bytes = 1 << 40, need - 256
    assert lib.kda_fwd(C.byref(a), None) == 1
    assert "workspace" in lib.kda_last_error().decode()


def test_workspace_sizes_scale_with_problem(lib):
    from gated_delta_rule_chunked_gb300 import _lib
    a = _fwd_args(total_tokens=32768, heads=96)
    chunks = 32768 // 64 + 1
    rec = 3 * 64 * 128 * 2 + 2 * 64 * 64 * 2 + 512
    assert lib.kda_fwd_workspace_size(C.byref(a)) >= chunks * 96 * rec
    # saved (bf16): chunk-start states, plus what the forward's prep writes for the backward:
    # the chunk record itself, fp32 A and T, and the Kt tile
    per = 128 * 128 * 2 + 2 * 64 * 64 * 4 + rec + 64 * 128 * 2
    assert chunks * 96 * per <= lib.kda_saved_size(C.byref(a)) <= chunks * 96 * per + 5 * 256
    # backward workspace: the chunk-end state gradients dS^T (bf16 128 x 128 per chunk and head)
    b = _lib.BwdArgs()
    b.fwd = a
    dsb = chunks * 96 * 128 * 128 * 2
    assert dsb <= lib.kda_bwd_workspace_size(C.byref(b)) <= dsb + 4 * 256 + 8 * (1 + 1) + 4096


def test_bwd_fp32_workspace(lib):
    # fp32: `saved` holds the chunk-start states only; the backward's workspace takes the chunk-end
    # gradients dS, the recomputed records, A and T, and the per-chunk scratch of the chunk kernels
    from gated_delta_rule_chunked_gb300 import _lib
    a = _fwd_args(total_tokens=4096, heads=8, io_dtype=_lib.KDA_F32)
    n = (4096 // 64 + 1) * 8
    assert n * 128 * 128 * 4 <= lib.kda_saved_size(C.byref(a)) <= n * 128 * 128 * 4 + 256
    b = _lib.BwdArgs()
    b.fwd = a
    per = 128 * 128 * 4 + (3 * 64 * 128 + 2 * 64 * 64) * 4 + 512 + 2 * 64 * 64 * 4 + (2 * 64 * 64 + 128) * 4
    assert n * per <= lib.kda_bwd_workspace_size(C.byref(b)) <= n * per + 6 * 256 + 4096


def test_step_validation(lib):
    from gated_delta_rule_chunked_gb300 import _lib
    a = _lib.StepArgs()
    a.n_seqs, a.steps, a.heads, a.dk, a.dv, a.scale = 4, 9, 2, 128, 128, 1.0
    fake = 1 << 40
    a.q = a.k = a.v = a.g = a.beta = a.state = a.o = fake
    assert lib.kda_step(C.byref(a), None) == 1     # steps > 8
    a.steps, a.dk = 4, 96
    assert lib.kda_step(C.byref(a), None) == 2
    a.dk, a.state = 128, None
    assert lib.kda_step(C.byref(a), None) == 1


def test_conv_validation(lib):
    from gated_delta_rule_chunked_gb300 import _lib
    fake = 1 << 40
    a = _lib.ConvArgs()
    a.n_seqs, a.total_tokens, a.channels, a.width, a.activation = 2, 64, 256, 4, _lib.KDA_ACT_SILU
    a.x = a.weight = a.y = a.state_in = fake
    a.width = 5
    assert lib.kda_conv_fwd(C.byref(a), None) == 2     # width > 4
    a.width, a.channels = 4, 100
    assert lib.kda_conv_fwd(C.byref(a), None) == 2     # channels not a multiple of 8
    a.channels, a.activation = 256, 7
    assert lib.kda_conv_fwd(C.byref(a), None) == 1
    a.activation, a.total_tokens = _lib.KDA_ACT_SILU, 63
    assert lib.kda_conv_fwd(C.byref(a), None) == 1     # 63 tokens do not split into 2 equal sequences
    a.total_tokens, a.state_out = 64, fake + 16         # overlaps state_in
    assert lib.kda_conv_fwd(C.byref(a), None) == 1
    a.state_out, a.x = None, fake + 4
    assert lib.kda_conv_fwd(C.byref(a), None) == 1     # misaligned x
    b = _lib.ConvBwdArgs()
    b.fwd = a
    b.fwd.x = fake
    b.dy, b.dx, b.dweight = fake, fake, fake
    assert lib.kda_conv_bwd(C.byref(b), None) == 1     # no workspace
    s = _lib.ConvStepArgs()
    s.n_seqs, s.steps, s.channels, s.width = 4, 9, 256, 4
    s.x = s.weight = s.state = s.y = fake
    assert lib.kda_conv_step(C.byref(s), None) == 1    # steps > 8
    s.steps, s.state = 4, None
    assert lib.kda_conv_step(C.byref(s), None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    from gated_delta_rule_chunked_gb300 import _lib
    saved = _lib._lib
    try:
        _lib._lib = None
        with pytest.raises(ImportError):
            _lib.load(str(tmp_path / "missing.so"))
    finally:
        _lib._lib = saved


def test_fwd_wait_fields_validation(lib):
    from gated_delta_rule_chunked_gb300 import _lib
    assert lib.kda_fwd(C.byref(_fwd_args(wait_limit_ns=-1)), None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd(C.byref(_fwd_args(debug_starve=1, io_dtype=_lib.KDA_F32)), None) == _lib.KDA_ERR_UNSUPPORTED


def _cp_args(n_segments=4, **over):
    from gated_delta_rule_chunked_gb300 import _lib
    c = _lib.FwdCpArgs()
    c.fwd = _fwd_args(**over)
    c.n_segments = n_segments
    return c


def test_fwd_cp_validation_and_workspace(lib):
    from gated_delta_rule_chunked_gb300 import _lib
    c = _cp_args()
    need = lib.kda_fwd_cp_workspace_size(C.byref(c))
    # three [N P][H][128][128] fp32 state arrays at least (N = 1, P = 4, H = 2)
    assert need >= 3 * 4 * 2 * 128 * 128 * 4
    assert lib.kda_fwd_cp_workspace_size(C.byref(_cp_args(n_segments=8))) > need
    assert lib.kda_fwd_cp(C.byref(c), None) == _lib.KDA_ERR_INVALID_ARG          # no workspace
    c.workspace, c.workspace_bytes = 1 << 40, need - 256
    assert lib.kda_fwd_cp(C.byref(c), None) == _lib.KDA_ERR_INVALID_ARG          # too small
    assert lib.kda_fwd_cp(C.byref(_cp_args(n_segments=0)), None) == _lib.KDA_ERR_INVALID_ARG
    # fp32 I/O is supported: its workspace holds fp32 records (larger), and a call still needs one
    assert lib.kda_fwd_cp_workspace_size(C.byref(_cp_args(io_dtype=_lib.KDA_F32))) > need
    assert lib.kda_fwd_cp(C.byref(_cp_args(io_dtype=_lib.KDA_F32)), None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_fwd_cp(C.byref(_cp_args(saved=1 << 40)), None) == _lib.KDA_ERR_UNSUPPORTED
    assert lib.kda_fwd_cp(C.byref(_cp_args(h0_identity=1)), None) == _lib.KDA_ERR_UNSUPPORTED
    assert lib.kda_fwd_cp(C.byref(_cp_args(v=None)), None) == _lib.KDA_ERR_INVALID_ARG   # v required
    # the caller's fwd.workspace is ignored: a misaligned one does not fail the size query
    assert lib.kda_fwd_cp_workspace_size(C.byref(_cp_args(workspace=3))) == need
