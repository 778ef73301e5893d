"""Seeded synthetic inputs for the KDA training forward + backward.

This module holds no arithmetic of the method: it only draws random tensors.
Both the CUDA path's tests/benchmark and the FP64 oracle are fed from here.

Recipe (one ``torch.Generator('cpu')`` per workload, seeded, draws in this order):
  1. (mixed-length packed workloads only) lengths = randint(1, max_len + 1, (N,))
  2. q, k, v, g, beta: float32 randn, rounded to bfloat16 (round-to-nearest-even)
  3. A_log = rand * ln(16)            (float32, [Hv])
  4. dt_bias = 0.1 * randn            (float32, [Hv, 128])
  5. h0 = 0.05 * randn                (float32, [N, Hv, 128, 128], value-first)
  6. do = bfloat16(randn)             (same shape as v)
  7. dfinal_state = 0.05 * randn      (float32, same shape as h0)
The distributions are those of the five named workloads below; the draw order
is this module's choice (the workloads fix distributions and seeds only).

Inference gate modes (``precomputed_gate_inputs``, a generator of its own):
a log-space gate g = bfloat16(-5 * rand), in [-5, 0], and an already
sigmoided beta = bfloat16(rand), in [0, 1].
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # physical batch (1 for packed)
    T: int            # tokens per batch row (total tokens for packed)
    hqk: int
    hv: int
    seed: int
    packed: bool
    lengths: tuple | None = None  # packed sequence lengths (fixed lists)
    mixed_n: int = 0              # packed: number of sequences with random lengths
    mixed_max: int = 0            # packed: lengths ~ U[1, mixed_max]

    @property
    def token_heads(self) -> int:
        return self.total_tokens_hint * self.hv

    @property
    def total_tokens_hint(self) -> int:
        if self.mixed_n:
            return sum(mixed_lengths(self.seed, self.mixed_n, self.mixed_max))
        return self.B * self.T


def mixed_lengths(seed: int, n: int, max_len: int) -> list[int]:
    gen = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(1, max_len + 1, (n,), generator=gen).tolist()


WORKLOADS = {
    "fixed_b1_t64_h2": Workload("fixed_b1_t64_h2", 1, 64, 2, 2, 0, False),
    "fixed_b2_t1024_h32": Workload("fixed_b2_t1024_h32", 2, 1024, 32, 32, 1, False),
    "fixed_b4_t2048_hqk16_hv32": Workload("fixed_b4_t2048_hqk16_hv32", 4, 2048, 16, 32, 2, False),
    "packed_8x1024_h96": Workload("packed_8x1024_h96", 1, 8192, 96, 96, 3, True,
                                  lengths=(1024,) * 8),
    "packed_24mixed_hqk8_hv64": Workload("packed_24mixed_hqk8_hv64", 1, 0, 8, 64, 4, True,
                                         mixed_n=24, mixed_max=4000),
    # half of the packed 8 x 1024 workload, for profiler captures (a few GB on the device)
    "packed_4x1024_h96": Workload("packed_4x1024_h96", 1, 4096, 96, 96, 5, True, lengths=(1024,) * 4),
}


def _bf16_randn(gen, shape):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(B: int, T: int, hqk: int, hv: int, seed: int, lengths=None,
                mixed=None, dim: int = DIM) -> dict:
    """Draw one problem. Fixed layout when ``lengths`` and ``mixed`` are None;
    packed (B must be 1) with the given ``lengths`` list, or with ``mixed=(n,
    max_len)`` random lengths drawn first from the same generator."""
    gen = torch.Generator("cpu").manual_seed(seed)
    if mixed is not None:
        n, max_len = mixed
        lengths = torch.randint(1, max_len + 1, (n,), generator=gen).tolist()
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        B, T = 1, sum(lengths)
        cu = torch.tensor([0] + list(_cumsum(lengths)), dtype=torch.int64)
        nseq = len(lengths)
    else:
        cu = None
        nseq = B
    q = _bf16_randn(gen, (B, T, hqk, dim))
    k = _bf16_randn(gen, (B, T, hqk, dim))
    v = _bf16_randn(gen, (B, T, hv, dim))
    g = _bf16_randn(gen, (B, T, hv, dim))
    beta = _bf16_randn(gen, (B, T, hv))
    A_log = torch.rand((hv,), generator=gen, dtype=torch.float32) * math.log(16.0)
    dt_bias = 0.1 * torch.randn((hv, dim), generator=gen, dtype=torch.float32)
    h0 = 0.05 * torch.randn((nseq, hv, dim, dim), generator=gen, dtype=torch.float32)
    do = _bf16_randn(gen, (B, T, hv, dim))
    dfinal_state = 0.05 * torch.randn((nseq, hv, dim, dim), generator=gen, dtype=torch.float32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias, h0=h0, do=do,
                dfinal_state=dfinal_state, cu_seqlens=cu)


def precomputed_gate_inputs(x: dict, seed: int) -> dict:
    """Copy of ``x`` whose g is drawn as a log-space gate in [-5, 0] and whose
    beta is drawn as a learning rate in [0, 1] (same shapes, bfloat16)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    y = dict(x)
    y["g"] = (-5.0 * torch.rand(x["g"].shape, generator=gen, dtype=torch.float32)).to(torch.bfloat16)
    y["beta"] = torch.rand(x["beta"].shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return y


def _cumsum(xs):
    s = 0
    for x in xs:
        s += x
        yield s


def workload_inputs(name: str) -> dict:
    w = WORKLOADS[name]
    if w.mixed_n:
        return make_inputs(1, 0, w.hqk, w.hv, w.seed, mixed=(w.mixed_n, w.mixed_max))
    return make_inputs(w.B, w.T, w.hqk, w.hv, w.seed, lengths=w.lengths)
