"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (fp32 outputs): |gpu - oracle| <= 1e-7 + 1e-6 * |oracle|, against the
oracle's double-precision value. Outputs stored in bf16 (probs for bf16 logits)
must be a correct bf16 rounding of a value within that fp32 tolerance: their
bound adds half a bf16 ulp of the oracle value. Indices, routing maps and the
sorted layout must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

RTOL = 1e-6
ATOL = 1e-7


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy()


def assert_close(gpu, ref, what: str, rtol: float = RTOL, atol: float = ATOL):
    g = np.asarray(to_np(gpu) if isinstance(gpu, torch.Tensor) else gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    bound = atol + rtol * np.abs(r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={g[i]!r} oracle={r[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")


def assert_bf16_close(gpu_bf16, ref, what: str):
    g = np.asarray(to_np(gpu_bf16), dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    mag = np.abs(r)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(mag > 0, mag, 1.0)))
    half_ulp = np.where(mag > 0, 2.0 ** (e - 8), 0.0)
    bound = half_ulp + ATOL + RTOL * mag
    err = np.abs(g - r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} bf16 values outside half an ulp; worst at {i}: "
                             f"gpu={g[i]!r} oracle={r[i]!r}")


def assert_equal(gpu, ref, what: str):
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if not np.array_equal(g, r):
        bad = np.argwhere(g != r)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches; first at {i}: gpu={g[i]!r} oracle={r[i]!r}")


def sample_rows(T: int, n: int, seed: int = 5) -> np.ndarray:
    """Sorted row indices: the first, the last and n-2 seeded random ones."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    rows.update({0, T - 1})
    return np.array(sorted(rows))


# (label, rows with a near tie, rows) of every parity case that noted them;
# conftest prints them at the end of the run
NEAR_TIES: list = []


def note_near_ties(orc, what: str, x, k_r: int, score_fn: int, bias=None, ulps: float = 4.0) -> int:
    """Records how many of these token rows have the last key taken and the
    first key left out within `ulps` fp32 ulps (keys in double, by the oracle).
    Informational: those are the rows where another rounding of the keys could
    change the selection, so they are where bit-exact agreement says the most."""
    xf = x.float().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float32)
    b = None if bias is None else (bias.float().numpy() if isinstance(bias, torch.Tensor) else bias)
    gaps = orc.near_tie_gaps(xf, k_r, score_fn, b)
    n = int(((gaps >= 0) & (gaps < ulps)).sum())
    NEAR_TIES.append((what, n, len(gaps)))
    return n
