"""Seeded synthetic inputs for the block-scaled int8 GEMM.

This module holds recipes for random fp32 matrices and nothing of the
method's arithmetic: no scales, no rounding, no products.  The tests feed the
same tensors to the CUDA library and to the CPU oracle, and the benchmark
draws its workload from here.  Every tensor is built on the CPU with a
seeded ``torch.Generator`` and is float32, row-major and contiguous.

Workloads (shapes are GPT-2-small-shaped only; no data or weights exist):

* ``square256``      256 x 256 x 256, A and B ~ N(0, 1), seed 0, no ReLU;
  plus 64 tiny shapes (M, N, K) drawn uniformly from 1..17 (seed 1000 + i).
* ``gpt2_linears``   M = 8192 tokens: QKV (K 768 -> N 2304), fc (768 -> 3072,
  fused ReLU), proj (3072 -> 768); activations ~ N(0, 1) with 0.1% of the
  entries (a seeded draw of positions) multiplied by 20; weights ~ N(0, 0.02).
* ``lm_head``        8192 x 50304 x 768, activations ~ N(0, 1), weights
  ~ N(0, 0.02); plus the 1024^3 probe GEMM (its inputs come from the probe's
  own generator, not from here).
* ``train_trio``     M = 8192, K = 768, N = 3072: forward X.W, grad-input
  dY.W^T, grad-weight X^T.dY; X ~ N(0, 1), W ~ N(0, 0.02), dY ~ N(0, 1e-3).
* ``squares``        4096^3, 8192^3, 16384^3 ~ U(-1, 1); ragged
  4097 x 12289 x 8191 ~ U(-1, 1); adversarial value mixes (see
  ``adversarial``).
"""
from __future__ import annotations

import math

import torch

__all__ = ["normal", "uniform", "gpt2_activations", "gpt2_weights", "tiny_shapes",
           "adversarial", "GPT2_LINEARS", "TRAIN_TRIO", "SQUARES", "RAGGED",
           "LM_HEAD", "PROBE_SHAPE", "ADVERSARIAL_KINDS", "LARGE_GEMMS",
           "large_gemm_inputs", "gpt2_linear_inputs"]

# (name, M, N, K, relu, seed)
GPT2_LINEARS = [
    ("qkv", 8192, 2304, 768, False, 1),
    ("fc", 8192, 3072, 768, True, 2),
    ("proj", 8192, 768, 3072, False, 3),
]
LM_HEAD = ("lm_head", 8192, 50304, 768, False, 4)
PROBE_SHAPE = (1024, 1024, 1024)
# (name, M, N, K, transA, transB): A_stored, B_stored as named in train_trio()
TRAIN_TRIO = [
    ("fwd", 8192, 3072, 768, False, False),
    ("dgrad", 8192, 768, 3072, False, True),
    ("wgrad", 768, 3072, 8192, True, False),
]
SQUARES = [(4096, 6), (8192, 7), (16384, 8)]
RAGGED = (4097, 12289, 8191, 9)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def uniform(shape, lo: float, hi: float, seed: int) -> torch.Tensor:
    x = torch.rand(*shape, generator=_gen(seed), dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def gpt2_activations(M: int, K: int, seed: int, outlier_frac: float = 1e-3,
                     outlier_gain: float = 20.0) -> torch.Tensor:
    """N(0, 1) activations with a seeded 0.1% of the entries scaled by 20."""
    g = _gen(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        idx = torch.randperm(M * K, generator=g)[:n_out]
        x.view(-1)[idx] *= outlier_gain
    return x


def gpt2_weights(K: int, N: int, seed: int, std: float = 0.02) -> torch.Tensor:
    return normal((K, N), std, seed + 7919)


def tiny_shapes(count: int = 64, base_seed: int = 1000):
    """(M, N, K, seed) for `count` tiny shapes with each size in 1..17."""
    out = []
    for i in range(count):
        g = _gen(base_seed + i)
        m, n, k = (int(v) for v in torch.randint(1, 18, (3,), generator=g))
        out.append((m, n, k, base_seed + i))
    return out


def gpt2_linear_inputs(name: str):
    """(A, B, relu) for one of the three GPT-2 linears."""
    for nm, M, N, K, relu, seed in GPT2_LINEARS:
        if nm == name:
            return gpt2_activations(M, K, seed), gpt2_weights(K, N, seed), relu
    raise KeyError(name)


def train_trio(M: int = 8192, K: int = 768, N: int = 3072, seed: int = 5):
    """X (M x K) ~ N(0,1), W (K x N) ~ N(0, 0.02), dY (M x N) ~ N(0, 1e-3)."""
    X = normal((M, K), 1.0, seed)
    W = normal((K, N), 0.02, seed + 1)
    dY = normal((M, N), 1e-3, seed + 2)
    return X, W, dY


# Row (or column) kinds of the adversarial mix.
ADVERSARIAL_KINDS = (
    "zero",          # all +0: the 1e-8 scale floor
    "neg_zero",      # all -0
    "ties",          # max = 127 * 2^e and x = (k + 1/2) * 2^e: exact quantize ties
    "subnormal",     # only subnormal values
    "subnormal_mix", # normal values with subnormals between them
    "huge",          # magnitude 1e30 (outputs overflow to +-Inf with a huge column)
    "tiny",          # magnitude 1e-30 (floored scale, every value quantizes to 0)
    "neg_max",       # the absmax is attained by a negative value only
    "spike",         # one large value, the rest tiny
)


def _adversarial_vector(kind: str, n: int, g: torch.Generator) -> torch.Tensor:
    u = torch.rand(n, generator=g, dtype=torch.float32) * 2 - 1
    if kind == "zero":
        return torch.zeros(n)
    if kind == "neg_zero":
        return torch.full((n,), -0.0)
    if kind == "ties":
        e = int(torch.randint(-20, 21, (1,), generator=g))
        k = torch.randint(-127, 127, (n,), generator=g).to(torch.float32)
        v = (k + 0.5) * (2.0 ** e)
        pos = int(torch.randint(0, n, (1,), generator=g))
        v[pos] = 127.0 * (2.0 ** e) * (1 if pos % 2 == 0 else -1)
        return v
    if kind == "subnormal":
        bits = torch.randint(1, 1 << 23, (n,), generator=g, dtype=torch.int64)
        sign = torch.randint(0, 2, (n,), generator=g, dtype=torch.int64) << 31
        return (bits | sign).to(torch.int32).view(torch.float32)
    if kind == "subnormal_mix":
        bits = torch.randint(1, 1 << 23, (n,), generator=g, dtype=torch.int64)
        sub = bits.to(torch.int32).view(torch.float32)
        mask = torch.rand(n, generator=g) < 0.5
        return torch.where(mask, u, sub)
    if kind == "huge":
        return u * 1e30
    if kind == "tiny":
        return u * 1e-30
    if kind == "neg_max":
        v = u * 0.5
        pos = int(torch.randint(0, n, (1,), generator=g))
        v[pos] = -3.0
        return v
    if kind == "spike":
        v = u * 1e-3
        pos = int(torch.randint(0, n, (1,), generator=g))
        v[pos] = 1e4
        return v
    raise KeyError(kind)


def adversarial(rows: int, length: int, seed: int, frac: float = 1.0 / 3.0,
                along_rows: bool = True) -> torch.Tensor:
    """A matrix whose vectors of one kind mix the adversarial cases.

    along_rows=True gives a rows x length matrix whose *rows* carry the kinds
    (for A); along_rows=False gives a length x rows matrix whose *columns*
    carry them (for B, where quantization runs down the columns).  A seeded
    `frac` of the vectors take the kinds in turn; the rest are U(-1, 1).
    """
    g = _gen(seed)
    out = torch.rand(rows, length, generator=g, dtype=torch.float32) * 2 - 1
    n_special = max(len(ADVERSARIAL_KINDS), int(math.ceil(frac * rows))) if rows else 0
    n_special = min(n_special, rows)
    picks = torch.randperm(rows, generator=g)[:n_special].tolist()
    for t, r in enumerate(picks):
        out[r] = _adversarial_vector(ADVERSARIAL_KINDS[t % len(ADVERSARIAL_KINDS)], length, g)
    return out if along_rows else out.t().contiguous()


# The large and adversarial GEMMs, (name, M, N, K, relu, seed): squares of
# U(-1, 1) values and the ragged shape with the adversarial mixes in A's rows
# and B's columns.  A takes `seed`, B `seed + 1`.
LARGE_GEMMS = [
    ("sq4096", 4096, 4096, 4096, False, SQUARES[0][1]),
    ("sq8192", 8192, 8192, 8192, False, SQUARES[1][1]),
    ("sq16384", 16384, 16384, 16384, False, SQUARES[2][1]),
    ("ragged_adversarial", RAGGED[0], RAGGED[1], RAGGED[2], False, RAGGED[3]),
]


def large_gemm_inputs(name: str):
    """(A, B, relu) for one of LARGE_GEMMS."""
    for nm, M, N, K, relu, seed in LARGE_GEMMS:
        if nm == name:
            if nm.startswith("sq"):
                return uniform((M, K), -1, 1, seed), uniform((K, N), -1, 1, seed + 1), relu
            return (adversarial(M, K, seed), adversarial(N, K, seed + 1, along_rows=False),
                    relu)
    raise KeyError(name)
