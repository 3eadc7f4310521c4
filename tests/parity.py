"""Shared comparison helpers for parity tests (GPU output vs the fp64 oracle).

Tolerances: max |diff| <= 1e-2 and mean |diff| <= 1e-3 over every compared
element (the stated bar for bf16 inputs with fp32 accumulation), plus a
relative L2 error <= 1e-2 so that long, nearly flat contexts (|out| ~ 0.01)
still have a meaningful check. bf16 rounding of the output alone contributes
a relative error of at most 2**-9 per element.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
REL_L2 = 1e-2


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 tensor to float64 numpy."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def stats(got: np.ndarray, want: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    d = np.abs(got - want)
    denom = float(np.linalg.norm(want.ravel()))
    rel = float(np.linalg.norm((got - want).ravel())) / denom if denom > 0 else float(np.linalg.norm(got.ravel()))
    return {
        "max_abs": float(d.max()) if d.size else 0.0,
        "mean_abs": float(d.mean()) if d.size else 0.0,
        "rel_l2": rel,
        "finite": bool(np.isfinite(got).all()),
        "n": int(d.size),
    }


def within(s: dict, max_abs=MAX_ABS, mean_abs=MEAN_ABS, rel_l2=REL_L2) -> bool:
    return s["finite"] and s["max_abs"] <= max_abs and s["mean_abs"] <= mean_abs and s["rel_l2"] <= rel_l2


def assert_close(got, want, what: str = "", **tol):
    s = stats(got, want)
    assert within(s, **tol), f"{what}: parity failed {s}"
    return s
