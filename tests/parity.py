"""Comparison metrics and gates for the GPU parity tests (test helper, not a test file).

Tolerances, from the arithmetic of each path:
  BF16 path vs FP64 attention: cosine >= 0.99999 and, elementwise,
      |O - O_ref| <= 2e-2 + 2^-7 * A|V|
  where A|V| = sum_j p_j |v_j| / sum_j p_j is the attention-weighted mean
  magnitude of V (the oracle evaluates it with |V| in place of V).  The
  kernel rounds every probability to BF16 before the P V product (relative
  error <= 2^-8 each, so at most 2^-8 A|V| on the output) and rounds O to BF16
  once more (<= 2^-8 |O| <= 2^-8 A|V|); 2e-2 is the absolute tolerance the
  acceptance criteria state for everything else.  On rows dominated by a few
  x8 outlier tokens A|V| reaches ~30, where no BF16 kernel that rounds P can
  stay within an absolute 2e-2.  Where no such rows exist (N(0,1) inputs: the
  tiny, FLUX-1024, FLUX-2048 and HunyuanVideo workloads and the small cases)
  the stated bound itself, max |O - O_ref| <= 2e-2, is asserted as well
  (assert_bf16_raw); only the Wan-720p workload, with its x8 outlier tokens,
  relies on the derived bound alone.
  Sage path vs the exact value of its own format (FP64 attention on the
  prepared INT8 / e4m3 codes): cosine >= 0.999 and
      |O - O_fmt| <= 1e-3 + (2^-4 + 2^-8) * A|V|_fmt
  (e4m3 probabilities, relative error <= 2^-4 each, and the BF16 output).
  Sage path vs FP64 attention of the BF16 inputs (the acceptance criteria):
  cosine >= 0.995 and max |O - O_ref| <= 0.1, plus the band of the Sage op's
  own test plan (aiter pull request, Test Plan: atol 0.3, rtol 0.25, at most
  0.5 % of elements outside, cosine >= 0.998, median row cosine >= 0.99).
"""
from __future__ import annotations

import numpy as np
import torch


def metrics(out, ref, bound_scale=None, a=0.0, b=0.0) -> dict:
    o = out.double().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    o2 = o.reshape(-1, o.shape[-1])
    r2 = r.reshape(-1, r.shape[-1])
    d = np.abs(o2 - r2)
    cos = float((o2 * r2).sum() / (np.linalg.norm(o2) * np.linalg.norm(r2) + 1e-300))
    rc = (o2 * r2).sum(1) / (np.linalg.norm(o2, axis=1) * np.linalg.norm(r2, axis=1) + 1e-300)
    m = dict(max_abs=float(d.max()), cos=cos, median_row_cos=float(np.median(rc)), min_row_cos=float(rc.min()),
             rel_l2=float(np.linalg.norm(o2 - r2) / (np.linalg.norm(r2) + 1e-300)),
             band_fail=float(np.mean(d > 0.3 + 0.25 * np.abs(r2))), nan=bool(np.isnan(o2).any()))
    if bound_scale is not None:
        s = np.asarray(bound_scale, dtype=np.float64).reshape(d.shape)
        m["bound_ratio"] = float((d / (a + b * s)).max())   # <= 1 passes
    return m


def assert_bf16_gate(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["cos"] >= 0.99999, f"{what}: cosine {m}"
    assert m["bound_ratio"] <= 1.0, f"{what}: error above 2e-2 + 2^-7 A|V| {m}"


def assert_bf16_raw(m: dict, what: str = ""):
    """The BF16 path's stated acceptance bound, max-abs <= 2e-2 against FP64, for inputs
    without outlier-dominated rows."""
    assert m["max_abs"] <= 2e-2, f"{what}: raw max-abs above 2e-2 {m}"


def assert_sage_format_gate(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["cos"] >= 0.999, f"{what}: cosine vs format-exact {m}"
    assert m["bound_ratio"] <= 1.0, f"{what}: error above 1e-3 + (2^-4 + 2^-8) A|V| {m}"


def assert_sage_exact_gate(m: dict, what: str = ""):
    assert not m["nan"], f"{what}: NaN in output {m}"
    assert m["cos"] >= 0.995, f"{what}: cosine {m}"
    assert m["max_abs"] <= 0.1, f"{what}: max-abs {m}"
    assert m["band_fail"] <= 0.005 and m["cos"] >= 0.998 and m["median_row_cos"] >= 0.99, f"{what}: band {m}"


BF16_A, BF16_B = 2e-2, 2.0 ** -7
SAGE_A, SAGE_B = 1e-3, 2.0 ** -4 + 2.0 ** -8


def gather_rows(o: torch.Tensor, rows: torch.Tensor) -> np.ndarray:
    """o: [B, S, H, D] (device or host), rows: int64 [n, 3] of (b, s, h) -> [n, D] float64."""
    r = rows.to(o.device)
    return o[r[:, 0], r[:, 1], r[:, 2]].double().cpu().numpy()
