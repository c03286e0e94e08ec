"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds random-number plumbing only, none of the attention
arithmetic.  Values are drawn on the CPU with ``torch.Generator`` in float32,
then rounded once to the working dtype; both the CUDA path and the CPU oracle
read those same rounded values.

Streams (independent generators, one per tensor, after the flaxattention
README's separate PRNG keys for key, query and value in "Example usage"):
k <- seed, q <- seed+1, v <- seed+2, dout <- seed+3, key_mask <- seed+4,
sampled query rows <- seed+5.  The default seed is 42, the seed that the
flash-attention-jax accuracy check uses ("2. Verify attention implementation").
"""

from __future__ import annotations

import torch

SEED = 42

_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
           "fp32": torch.float32, "fp16": torch.float16}


def torch_dtype(name):
    return _DTYPES[name] if isinstance(name, str) else name


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn(shape, seed: int, dtype="f32") -> torch.Tensor:
    """N(0, 1) in float32 from its own generator, then rounded to ``dtype``."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32).to(torch_dtype(dtype))


def key_mask(B: int, Skv: int, seed: int) -> torch.Tensor:
    """Uniform {0, 1} integers of shape (B, Skv), uint8 (1 = attend)."""
    return torch.randint(0, 2, (B, Skv), generator=_gen(seed), dtype=torch.int64).to(torch.uint8)


def make_case(B, H, Sq, Skv, D, dtype="bf16", seed: int = SEED, with_key_mask=False,
              dout="randn"):
    """q, k, v, dout (and optionally key_mask) on the CPU, BHSD contiguous."""
    out = {
        "k": randn((B, H, Skv, D), seed, dtype),
        "q": randn((B, H, Sq, D), seed + 1, dtype),
        "v": randn((B, H, Skv, D), seed + 2, dtype),
    }
    if dout == "ones":
        out["dout"] = torch.ones((B, H, Sq, D), dtype=torch_dtype(dtype))
    elif dout == "randn":
        out["dout"] = randn((B, H, Sq, D), seed + 3, dtype)
    elif dout is not None:
        raise ValueError(dout)
    out["key_mask"] = key_mask(B, Skv, seed + 4) if with_key_mask else None
    return out


def sample_rows(Sq: int, n: int, seed: int = SEED + 5) -> torch.Tensor:
    """n distinct query rows, always including 0 and Sq-1, sorted (int64)."""
    if n >= Sq:
        return torch.arange(Sq, dtype=torch.int64)
    g = _gen(seed)
    rest = torch.randperm(Sq - 2, generator=g)[: max(0, n - 2)].to(torch.int64) + 1
    rows = torch.cat([torch.tensor([0, Sq - 1], dtype=torch.int64), rest])
    return torch.sort(rows).values
