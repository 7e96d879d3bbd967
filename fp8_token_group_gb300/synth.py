"""Seeded synthetic inputs for the quantizer's workloads.

This module holds no quantization arithmetic: it only draws random activations
(and masked-row counts) with fixed seeds, so that the CUDA path, the CPU oracle
and the benchmark all see bit-identical inputs.  Every tensor is generated on
the CPU with ``torch.Generator('cpu')`` and returned on the CPU.

Workloads (shapes and distributions follow the pages' test and benchmark
shapes; all data is synthetic, no model weights or datasets are involved):

* ``flat_small``     bf16 [64, 4096] ~ N(0,1), seed 0.
* ``flat_outliers``  bf16 [4096, 7168] ~ N(0,1), seed 0; 0.1% of elements x100
                     (Bernoulli(1e-3), seed 1); 1% of 128-groups set to zero
                     (Bernoulli(1e-2) over [4096, 56], seed 2).
* ``silu_flat``      bf16 [8192, 2*2048] gate|up ~ N(0,1), seed 0.
* ``masked_silu``    bf16 [32, 384, 2*4096] ~ N(0,1), seed 0; masked_m[e]
                     uniform in [0, 384] (seed 0).
* ``sweep``          N(0,1) rows, with every row r % 4 == 3 replaced by integers
                     drawn uniformly from [-8, 8]; seed = case index.
"""
from __future__ import annotations

import itertools

import torch

__all__ = [
    "normal", "flat_small", "flat_outliers", "silu_flat", "masked_silu", "masked_counts",
    "sweep_cases", "sweep_input", "bits_u16",
]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, dtype=torch.bfloat16, seed: int = 0) -> torch.Tensor:
    """N(0,1) in fp32, rounded to ``dtype``."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32).to(dtype)


def flat_small(dtype=torch.bfloat16) -> torch.Tensor:
    return normal((64, 4096), dtype, seed=0)


def flat_outliers(tokens: int = 4096, hidden: int = 7168, group: int = 128,
                  dtype=torch.bfloat16) -> torch.Tensor:
    x = torch.randn((tokens, hidden), generator=_gen(0), dtype=torch.float32)
    spikes = torch.rand((tokens, hidden), generator=_gen(1)) < 1e-3
    x = torch.where(spikes, x * 100.0, x)
    dead = torch.rand((tokens, hidden // group), generator=_gen(2)) < 1e-2
    x = x.view(tokens, hidden // group, group).masked_fill(dead.unsqueeze(-1), 0.0)
    return x.view(tokens, hidden).to(dtype)


def silu_flat(tokens: int = 8192, hidden: int = 2048, dtype=torch.bfloat16) -> torch.Tensor:
    return normal((tokens, 2 * hidden), dtype, seed=0)


def masked_counts(experts: int = 32, tokens_pad: int = 384, seed: int = 0) -> torch.Tensor:
    """int32[E], each uniform in [0, tokens_pad]."""
    return torch.randint(0, tokens_pad + 1, (experts,), generator=_gen(seed), dtype=torch.int32)


def masked_silu(experts: int = 32, tokens_pad: int = 384, hidden: int = 4096,
                dtype=torch.bfloat16):
    x = normal((experts, tokens_pad, 2 * hidden), dtype, seed=0)
    return x, masked_counts(experts, tokens_pad, seed=0)


SWEEP_TOKENS = (1, 7, 64, 333, 4096, 32768)
SWEEP_HIDDEN = (128, 2048, 4096, 7168)
SWEEP_DTYPES = (torch.float16, torch.bfloat16)
SWEEP_GROUPS = (16, 32, 64, 128)
SWEEP_OUTS = ("e4m3", "int8")


def masked_decode(experts: int = 32, tokens_pad: int = 384, hidden: int = 4096, live: int = 1,
                  dtype=torch.bfloat16):
    """Decode-sized masked batch: the [E, tokens_pad, 2*hidden] buffer of the masked
    workload with `live` rows in every expert."""
    x = normal((experts, tokens_pad, 2 * hidden), dtype, seed=0)
    return x, torch.full((experts,), live, dtype=torch.int32)


def sweep_cases():
    """All (index, tokens, hidden, dtype, group, out) tuples of the shape sweep."""
    prod = itertools.product(SWEEP_TOKENS, SWEEP_HIDDEN, SWEEP_DTYPES, SWEEP_GROUPS, SWEEP_OUTS)
    return [(i, *c) for i, c in enumerate(prod)]


def sweep_input(index: int, tokens: int, hidden: int, dtype, rows=None) -> torch.Tensor:
    """The sweep case's input; ``rows`` optionally selects a subset of rows.

    Rows are generated in full and then sliced, so a row subset is bit-identical
    to the same rows of the full input.
    """
    g = _gen(index)
    x = torch.randn((tokens, hidden), generator=g, dtype=torch.float32)
    ints = torch.randint(-8, 9, (tokens, hidden), generator=g).to(torch.float32)
    int_rows = (torch.arange(tokens) % 4 == 3).unsqueeze(1)
    x = torch.where(int_rows, ints, x).to(dtype)
    return x if rows is None else x[rows]


def bits_u16(t: torch.Tensor):
    """The bit patterns of a CPU 16-bit tensor as a C-contiguous numpy uint16 array."""
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.contiguous().view(torch.int16).numpy().view("uint16")
