"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
the float64 oracle on the same seeded inputs, and compare.

Tolerances (written here once, used by every parity test):
  float32 inputs: max |err| <= 1e-4 on out and lse, <= 1e-3 on dq, dk, dv, at
                  every shape, never scaled.
  16-bit inputs:  max |err| <= 2e-2 and mean |err| <= 2e-3 on out, dq, dk, dv;
                  lse max |err| <= 2e-2 (lse is float32 on both sides).
Where a 16-bit result is large, the absolute bound becomes relative: the
result is stored in the 16-bit input type, whose own rounding step grows with
the value (bf16 rounds values in [2, 4) to steps of 2^-6 = 1.6e-2, values in
[4, 8) to 3.1e-2).  So
  out   (a convex combination of rows of v, |out| <= max |v|): bounds x
        max(1, max |ref| / 4): plain absolute bounds while |ref| <= 4;
  grads (no such bound; the small shapes reach |dq| ~ 4): bounds x
        max(1, max |ref|);
  lse   is float32 and is never scaled.
Every comparison records its achieved max and mean error against its bound;
the session prints the tightest margins per (dtype, tensor kind), and writes
the full list to the file named by ATTN_PARITY_LOG when that is set.
Masking is exact: the visited-tile map must equal the oracle's skip set, and
a row with no kept key must give out = 0 and lse = -inf bit for bit.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.attention as OR  # noqa: F401  (re-exported for the tests)
from exact_attention_59_gb300 import inputs as IN

TOL = {
    "f32": dict(o_max=1e-4, lse_max=1e-4, g_max=1e-3, o_mean=None, g_mean=None),
    "f16": dict(o_max=2e-2, lse_max=2e-2, g_max=2e-2, o_mean=2e-3, g_mean=2e-3),
    "bf16": dict(o_max=2e-2, lse_max=2e-2, g_max=2e-2, o_mean=2e-3, g_mean=2e-3),
}

# (name, dtype, kind, max err, max bound, mean err, mean bound) of every comparison
RECORDS: list[tuple] = []


def f64(t):
    return t.detach().float().cpu().double().numpy()


def bound_factor(dtype, kind, ref):
    """Multiplier of the absolute bounds (see the module docstring)."""
    if dtype not in ("f16", "bf16") or ref.size == 0:
        return 1.0
    m = float(np.abs(ref).max())
    if kind == "out":
        return max(1.0, m / 4.0)
    if kind == "grad":
        return max(1.0, m)
    return 1.0


def compare(name, got, ref, max_tol, mean_tol=None, mask=None, dtype=None, kind=None, relative=True):
    """max / mean |got - ref| against the bounds; ``dtype`` ("f32", "f16", "bf16")
    and ``kind`` ("out", "lse", "grad") select the 16-bit relative rule, which
    ``relative=False`` turns off (plain absolute bounds)."""
    g = np.asarray(got)
    r = np.asarray(ref)
    if mask is not None:
        g, r = g[mask], r[mask]
    f = bound_factor(dtype, kind, r) if relative else 1.0
    max_tol = max_tol * f
    mean_tol = None if mean_tol is None else mean_tol * f
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = np.abs(g - r)
    mx = float(err.max()) if err.size else 0.0
    mn = float(err.mean()) if err.size else 0.0
    RECORDS.append((name, dtype or "?", kind or name, mx, max_tol, mn, mean_tol))
    assert mx <= max_tol, f"{name}: max abs err {mx:.3e} > {max_tol:.3e}"
    if mean_tol is not None:
        assert mn <= mean_tol, f"{name}: mean abs err {mn:.3e} > {mean_tol:.3e}"
    return mx, mn


def margin_summary():
    """Lines: per (dtype, kind) the number of comparisons and the largest
    err / bound ratio seen, for max and mean errors."""
    worst = {}
    for name, dt, kind, mx, mtol, mn, ntol in RECORDS:
        key = (dt, kind)
        n, rmax, rmean = worst.get(key, (0, 0.0, 0.0))
        rmax = max(rmax, mx / mtol if mtol else 0.0)
        rmean = max(rmean, mn / ntol if ntol else 0.0)
        worst[key] = (n + 1, rmax, rmean)
    return [f"{dt:>4} {kind:<5} n={n:<4} worst max-err/bound {rmax:.3f}  worst mean-err/bound {rmean:.3f}"
            for (dt, kind), (n, rmax, rmean) in sorted(worst.items())]


def make_dev(B, H, Sq, Skv, D, dtype, key_mask=False, dout="randn", seed=IN.SEED):
    c = IN.make_case(B, H, Sq, Skv, D, dtype, seed=seed, with_key_mask=key_mask, dout=dout)
    dev = {k: (v.cuda() if v is not None else None) for k, v in c.items()}
    return c, dev


def guarded(shape, dtype, fill=float("nan"), canary=4096):
    """An output tensor filled with `fill`, followed by a canary region of 0x5A bytes."""
    n = int(np.prod(shape))
    esz = torch.empty((), dtype=dtype).element_size()
    extra = canary // esz
    buf = torch.full((n + extra,), fill, dtype=dtype, device="cuda")
    buf.view(torch.uint8)[n * esz:].fill_(0x5A)
    return buf, buf[:n].view(shape)


def canary_ok(buf, shape):
    n = int(np.prod(shape))
    esz = buf.element_size()
    tail = buf.view(torch.uint8)[n * esz:]
    return bool((tail == 0x5A).all().item())
