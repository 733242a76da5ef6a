"""Comparison metrics for the GPU parity tests (test helper, not a test file).

Tolerances (written in the tests that use them):
  BF16 path:  cosine >= 0.99999 and max |O - O_ref| <= 2e-2, where for
              |O_ref| > 1 the bound scales with |O_ref| (the kernel rounds O
              and P to BF16, whose step is relative: 2^-8 |x|; on rows of x8
              outlier tokens |O| reaches ~30 and no BF16 result is within an
              absolute 2e-2).  The raw max-abs is reported beside it.
  Sage path:  cosine >= 0.995 and max-abs <= 0.1 with the same scaling.
Secondary band (aiter pull request "gfx1201_sage_prepare /
gfx1201_sage_attention", Test Plan): atol 0.3, rtol 0.25 with at most 0.5 %
of elements outside, cosine >= 0.998 and median row cosine >= 0.99.
"""
from __future__ import annotations

import numpy as np
import torch


def metrics(out: torch.Tensor | np.ndarray, ref: np.ndarray) -> dict:
    o = out.double().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    o2 = o.reshape(-1, o.shape[-1])
    r2 = r.reshape(-1, r.shape[-1])
    d = np.abs(o2 - r2)
    scaled = d / np.maximum(1.0, np.abs(r2))
    cos = float((o2 * r2).sum() / (np.linalg.norm(o2) * np.linalg.norm(r2) + 1e-300))
    rc = (o2 * r2).sum(1) / (np.linalg.norm(o2, axis=1) * np.linalg.norm(r2, axis=1) + 1e-300)
    band_fail = float(np.mean(d > 0.3 + 0.25 * np.abs(r2)))
    return dict(max_abs=float(d.max()), max_scaled=float(scaled.max()), cos=cos, median_row_cos=float(np.median(rc)),
                min_row_cos=float(rc.min()), rel_l2=float(np.linalg.norm(o2 - r2) / (np.linalg.norm(r2) + 1e-300)),
                band_fail=band_fail, nan=bool(np.isnan(o2).any()))


def assert_bf16_gate(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["cos"] >= 0.99999, f"{what}: cosine {m}"
    assert m["max_scaled"] <= 2e-2, f"{what}: max error {m}"


def assert_sage_gate(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["cos"] >= 0.995, f"{what}: cosine {m}"
    assert m["max_scaled"] <= 0.1, f"{what}: max error {m}"
    # secondary band of the Sage op's own test plan
    assert m["band_fail"] <= 0.005 and m["cos"] >= 0.998 and m["median_row_cos"] >= 0.99, f"{what}: band {m}"


def gather_rows(o: torch.Tensor, rows: torch.Tensor) -> np.ndarray:
    """o: [B, S, H, D] (device or host), rows: int64 [n, 3] of (b, s, h) -> [n, D] float64."""
    r = rows.to(o.device)
    return o[r[:, 0], r[:, 1], r[:, 2]].double().cpu().numpy()
