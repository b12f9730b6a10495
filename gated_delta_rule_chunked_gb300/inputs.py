"""Seeded synthetic inputs for the KDA workloads.

This module is shared by the tests, the benchmark and the oracle checks. It holds
only the data recipe -- shapes, distributions, seeds and draw order -- and none of
the method's arithmetic, so the CUDA path and the oracle can both consume it
without sharing any computation.

Recipe (K3-shaped: 96 heads x 128 dims, from the KDA entry of the architecture
figure in "Kimi K3 模型结构（10）：RL 与服务中的状态管理"):

* q, k, v, dO ~ N(0, 1), drawn in fp32 and rounded to the I/O dtype;
* beta = sigmoid(N(0, 1)) per token and head (fp32);
* g = logsigmoid(N(3, 1)) per token, head and key channel (fp32, so g <= 0);
* initial states ~ N(0, 0.02) (0.02 is the standard deviation), fp32;
* packed variable-length batches: each sequence gets 1024 tokens plus one piece
  of a uniform random split (7 sorted uniform cut points) of the remainder;
* decode accept lengths ~ U{1..L}.

Draws always happen in the fixed order q, k, v, beta-logit, g-logit, dO, h0,
lengths, accept_len from one torch.Generator seeded per workload.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

D_HEAD = 128
CHUNK = 64


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "fwd", "fwdbwd" or "decode"
    io_dtype: str             # "bf16" or "f32"
    heads: int
    seq_lens: tuple = ()      # one entry per sequence (fwd / fwdbwd)
    varlen_total: int = 0     # >0: split this many tokens into varlen_seqs sequences
    varlen_seqs: int = 0
    varlen_min: int = 0
    h0: bool = False
    n_seqs: int = 0           # decode: independent sequences
    steps: int = 0            # decode: tokens per call
    seed: int = 0


# The five workloads of the KDA hot path, and a 128K-token point for the benchmark.
# Seeds are 1000 + the workload index.
WORKLOADS = {
    "fwd-f32-T512-H2": Workload("fwd-f32-T512-H2", "fwd", "f32", 2, seq_lens=(512,), seed=1000),
    "fwd-bf16-T4096-H96": Workload("fwd-bf16-T4096-H96", "fwd", "bf16", 96, seq_lens=(4096,), seed=1001),
    "fwdbwd-bf16-T32768-H96": Workload("fwdbwd-bf16-T32768-H96", "fwdbwd", "bf16", 96,
                                       seq_lens=(32768,), h0=True, seed=1002),
    "fwdbwd-bf16-varlen8-T131072-H96": Workload("fwdbwd-bf16-varlen8-T131072-H96", "fwdbwd", "bf16", 96,
                                                varlen_total=131072, varlen_seqs=8, varlen_min=1024,
                                                h0=True, seed=1003),
    "decode-bf16-N256-L4-H96": Workload("decode-bf16-N256-L4-H96", "decode", "bf16", 96,
                                        n_seqs=256, steps=4, h0=True, seed=1004),
    # the long end of the pages' 4K-128K sequence range, one sequence (benchmark only)
    "fwdbwd-bf16-T131072-H96": Workload("fwdbwd-bf16-T131072-H96", "fwdbwd", "bf16", 96,
                                        seq_lens=(131072,), h0=True, seed=1005),
}


@dataclass
class SeqBatch:
    """Inputs of a chunked (training) call, packed along tokens."""
    q: torch.Tensor           # [total, H, 128] io dtype
    k: torch.Tensor           # [total, H, 128] io dtype
    v: torch.Tensor           # [total, H, 128] io dtype
    beta: torch.Tensor        # [total, H] fp32
    g: torch.Tensor           # [total, H, 128] fp32
    cu_seqlens: torch.Tensor  # [N+1] int32
    h0: Optional[torch.Tensor] = None   # [N, H, 128, 128] fp32
    dO: Optional[torch.Tensor] = None   # [total, H, 128] io dtype
    meta: dict = field(default_factory=dict)

    @property
    def n_seqs(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def total(self) -> int:
        return self.q.shape[0]

    @property
    def heads(self) -> int:
        return self.q.shape[1]


@dataclass
class DecodeBatch:
    """Inputs of a decode / draft-verify call: L tokens for each of N sequences."""
    q: torch.Tensor           # [N, L, H, 128] io dtype
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor        # [N, L, H] fp32
    g: torch.Tensor           # [N, L, H, 128] fp32
    state: torch.Tensor       # [N, H, 128, 128] fp32
    accept_len: torch.Tensor  # [N] int32
    meta: dict = field(default_factory=dict)


def _dtype(io_dtype: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[io_dtype]


def _normal(gen, shape, device, std=1.0, mean=0.0):
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(mean=mean, std=std, generator=gen)
    return x


def varlen_split(total: int, n: int, min_len: int, gen: torch.Generator) -> list:
    """Lengths min_len + pieces of a uniform random split of the remainder."""
    rest = total - n * min_len
    if rest < 0:
        raise ValueError("total too small for the minimum length")
    cuts = torch.randint(0, rest + 1, (n - 1,), generator=gen).sort().values.tolist()
    edges = [0] + cuts + [rest]
    return [min_len + edges[i + 1] - edges[i] for i in range(n)]


def make_seq_batch(seq_lens, heads: int, io_dtype: str = "bf16", *, seed: int = 0,
                   h0: bool = False, grad: bool = False, device="cpu",
                   varlen: Optional[tuple] = None, d: int = D_HEAD,
                   beta_range: Optional[tuple] = None) -> SeqBatch:
    """Draw one packed batch. ``varlen=(total, n, min_len)`` draws the lengths from the seed."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens_gen = torch.Generator()          # lengths are always drawn on the host
    lens_gen.manual_seed(seed + 7919)
    if varlen is not None:
        seq_lens = varlen_split(*varlen, lens_gen)
    seq_lens = [int(x) for x in seq_lens]
    total = sum(seq_lens)
    dt = _dtype(io_dtype)
    q = _normal(gen, (total, heads, d), device).to(dt)
    k = _normal(gen, (total, heads, d), device).to(dt)
    v = _normal(gen, (total, heads, d), device).to(dt)
    beta = torch.sigmoid(_normal(gen, (total, heads), device))
    g = torch.nn.functional.logsigmoid(_normal(gen, (total, heads, d), device, mean=3.0))
    dO = _normal(gen, (total, heads, d), device).to(dt) if grad else None
    h = _normal(gen, (len(seq_lens), heads, d, d), device, std=0.02) if h0 else None
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(seq_lens, dtype=torch.int64).cumsum(0).to(torch.int32)
    return SeqBatch(q, k, v, beta, g, cu.to(device), h, dO,
                    meta={"seq_lens": seq_lens, "seed": seed, "io_dtype": io_dtype})


def make_decode_batch(n_seqs: int, steps: int, heads: int, io_dtype: str = "bf16", *,
                      seed: int = 0, device="cpu", d: int = D_HEAD) -> DecodeBatch:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = _dtype(io_dtype)
    shp = (n_seqs, steps, heads, d)
    q = _normal(gen, shp, device).to(dt)
    k = _normal(gen, shp, device).to(dt)
    v = _normal(gen, shp, device).to(dt)
    beta = torch.sigmoid(_normal(gen, (n_seqs, steps, heads), device))
    g = torch.nn.functional.logsigmoid(_normal(gen, shp, device, mean=3.0))
    state = _normal(gen, (n_seqs, heads, d, d), device, std=0.02)
    acc_gen = torch.Generator()
    acc_gen.manual_seed(seed + 104729)
    accept = torch.randint(1, steps + 1, (n_seqs,), generator=acc_gen, dtype=torch.int32)
    return DecodeBatch(q, k, v, beta, g, state, accept.to(device),
                       meta={"seed": seed, "io_dtype": io_dtype})


def make_workload(name: str, device="cpu", **over):
    """Build the inputs of one named workload (optionally overriding fields)."""
    w = WORKLOADS[name]
    if over:
        w = Workload(**{**w.__dict__, **over})
    if w.kind == "decode":
        return make_decode_batch(w.n_seqs, w.steps, w.heads, w.io_dtype, seed=w.seed, device=device)
    varlen = (w.varlen_total, w.varlen_seqs, w.varlen_min) if w.varlen_total else None
    return make_seq_batch(w.seq_lens, w.heads, w.io_dtype, seed=w.seed, h0=w.h0,
                          grad=(w.kind == "fwdbwd"), device=device, varlen=varlen)
