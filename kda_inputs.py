"""Seeded synthetic inputs for chunked KDA prefill.

This module is shared by the fp64 oracle and the CUDA path's tests and
benchmark. It draws random numbers and lays out tensors; it holds none of the
method's arithmetic (no decay, no state update, no chunking).

Workloads follow the shapes the pages speak of ("MoonEP / FlashKDA /
AgentENV" release note, section "MoE通信とアテンション": fixed-length and
varlen prefill at T=8192, head dim 128, 64 or 96 heads; K=V=128 only) plus a
tiny case and a long-context case. Recipe, per workload, with one CPU
``torch.Generator`` seeded with the workload's seed, drawing in this order:

1. varlen only: sequence lengths ``64 + m`` with ``m ~ Multinomial(T - 64*n,
   uniform over n bins)``, redrawn as a whole until no length is a multiple
   of 16;
2. q, k, v ~ N(0, 1) in fp32, shape [T, H, 128];
3. x_g ~ N(mu, 1) in fp32, [T, H, 128];
4. x_b ~ N(0, 1) in fp32, [T, H];
5. initial state ~ N(0, 0.02^2) (0.02 is the standard deviation), fp32
   [n_seqs, H, 128, 128], when the workload has one.

Then q and k are L2-normalised in fp32 over the 128 channels of each
(token, head) and rounded to bf16 (round to nearest even); v is rounded to
bf16; g = logsigmoid(x_g) (fp32, always <= 0); beta = sigmoid(x_b) (fp32, in
(0, 1)). Both sides of a parity test consume these exact values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

D = 128  # K = V = 128, the only head size the method supports


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    T: int                      # total tokens (all sequences packed)
    H: int
    n_seqs: int = 1
    varlen: bool = False        # True: packed sequences described by cu_seqlens
    init_state: bool = False
    mu: float = 3.0             # mean of the gate pre-activation
    seqlens: Optional[tuple] = None  # explicit lengths (overrides the draw)

    @property
    def tokens(self) -> int:
        return self.T


# The five workloads: the tiny case, the headline fixed-length case, more
# heads, varlen with initial states, and long context with stronger decay.
WORKLOADS = {
    "tiny_T64_H1": Workload("tiny_T64_H1", seed=0, T=64, H=1),
    "fixed_T8192_H64": Workload("fixed_T8192_H64", seed=1, T=8192, H=64),
    "fixed_T8192_H96": Workload("fixed_T8192_H96", seed=2, T=8192, H=96),
    "varlen16_T8192_H64": Workload("varlen16_T8192_H64", seed=3, T=8192, H=64, n_seqs=16,
                                   varlen=True, init_state=True),
    "long_T131072_H32": Workload("long_T131072_H32", seed=4, T=131072, H=32,
                                 init_state=True, mu=2.0),
}
WORKLOAD_ORDER = list(WORKLOADS)
HEADLINE = "fixed_T8192_H64"


def draw_varlen_lengths(gen: torch.Generator, total: int, n: int, min_len: int = 64) -> list:
    """Lengths ``min_len + Multinomial(total - n*min_len, uniform over n)``,
    redrawn until none is a multiple of 16 (every sequence ends in a partial
    chunk)."""
    spare = total - n * min_len
    if spare < 0:
        raise ValueError("total too small for n sequences of min_len")
    probs = torch.full((n,), 1.0 / n, dtype=torch.float64)
    for _ in range(10000):
        if spare > 0:
            picks = torch.multinomial(probs, spare, replacement=True, generator=gen)
            counts = torch.bincount(picks, minlength=n)
        else:
            counts = torch.zeros(n, dtype=torch.int64)
        lens = [min_len + int(c) for c in counts]
        if all(L % 16 != 0 for L in lens):
            return lens
    raise RuntimeError("could not draw lengths that avoid multiples of 16")


def _l2norm_bf16(x: torch.Tensor) -> torch.Tensor:
    n = torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-12)
    return (x / n).to(torch.bfloat16)


def make_inputs(w: Workload) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with q, k, v (bf16 [T, H, 128]), g (fp32 [T, H, 128]),
    beta (fp32 [T, H]), initial_state (fp32 [n_seqs, H, 128, 128] or None),
    cu_seqlens (int32 [n_seqs + 1]; always present, also for one sequence),
    seqlens (list of int), scale (float).
    """
    gen = torch.Generator().manual_seed(w.seed)
    if w.seqlens is not None:
        lens = list(w.seqlens)
        if sum(lens) != w.T or len(lens) != w.n_seqs:
            raise ValueError("seqlens disagree with T / n_seqs")
    elif w.varlen:
        lens = draw_varlen_lengths(gen, w.T, w.n_seqs)
    else:
        if w.T % w.n_seqs:
            raise ValueError("fixed-length workload needs T divisible by n_seqs")
        lens = [w.T // w.n_seqs] * w.n_seqs
    T, H = w.T, w.H
    q = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    k = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    v = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    xg = torch.randn(T, H, D, generator=gen, dtype=torch.float32) + w.mu
    xb = torch.randn(T, H, generator=gen, dtype=torch.float32)
    s0 = None
    if w.init_state:
        s0 = torch.randn(w.n_seqs, H, D, D, generator=gen, dtype=torch.float32) * 0.02
    q = _l2norm_bf16(q)
    k = _l2norm_bf16(k)
    v = v.to(torch.bfloat16)
    g = torch.nn.functional.logsigmoid(xg)
    beta = torch.sigmoid(xb)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, initial_state=s0, cu_seqlens=cu,
                seqlens=lens, scale=1.0 / math.sqrt(D))


def make_case(seqlens: Sequence[int], H: int, seed: int, init_state: bool = False,
              mu: float = 3.0) -> dict:
    """A small test case with explicit sequence lengths (zero allowed)."""
    lens = [int(L) for L in seqlens]
    w = Workload(f"case_{seed}", seed=seed, T=sum(lens), H=H, n_seqs=len(lens),
                 varlen=len(lens) > 1, init_state=init_state, mu=mu, seqlens=tuple(lens))
    return make_inputs(w)


def make_raw_case(seqlens: Sequence[int], H: int, seed: int, init_state: bool = False,
                  mu: float = 3.0) -> dict:
    """Like ``make_case`` but with raw projections, for the kernels' input
    preprocessing: q and k are N(0, 1) rows times a per-(token, head) factor
    drawn uniformly from [0.25, 4] (not normalised), rounded to bf16, and g
    holds the gate logits x ~ N(mu, 1) themselves. v, beta, the initial state
    and cu_seqlens are drawn as in ``make_inputs``."""
    lens = [int(L) for L in seqlens]
    T = sum(lens)
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    k = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    v = torch.randn(T, H, D, generator=gen, dtype=torch.float32)
    xg = torch.randn(T, H, D, generator=gen, dtype=torch.float32) + mu
    xb = torch.randn(T, H, generator=gen, dtype=torch.float32)
    s0 = None
    if init_state:
        s0 = torch.randn(len(lens), H, D, D, generator=gen, dtype=torch.float32) * 0.02
    fq = 0.25 + 3.75 * torch.rand(T, H, 1, generator=gen)
    fk = 0.25 + 3.75 * torch.rand(T, H, 1, generator=gen)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=(q * fq).to(torch.bfloat16), k=(k * fk).to(torch.bfloat16),
                v=v.to(torch.bfloat16), g=xg, beta=torch.sigmoid(xb), initial_state=s0,
                cu_seqlens=cu, seqlens=lens, scale=1.0 / math.sqrt(D))
