"""Tolerances and helpers for comparing the CUDA path with the CPU oracle.

Bars (fixed once here, used by every parity test):

* integer and index outputs (expert ids, counts, offsets, dispatch maps,
  gathered rows): bit-exact; dispatch rows are compared as a per-expert set
  because the order inside an expert is left open by the pages;
* FP32 outputs: every element within ``1e-4 * |ref| + 1e-6 * RMS(ref)`` and
  the largest error within ``1e-4 * max|ref|``;
* BF16 / F16 outputs: largest absolute error <= ``2e-2 * RMS(ref)``, with
  ``ref`` the unrounded float64 oracle result on the same rounded inputs;
* NaN positions must match exactly in every case; RMS is taken over the
  finite reference entries.
"""

from __future__ import annotations

import numpy as np
import torch

from mixture_experts_ffn_topk_gb300 import workloads as W

TORCH_TO_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def oracle_f64(a: np.ndarray, dt: str) -> np.ndarray:
    """Oracle-storage array (raw 16-bit words for bf16/f16) -> float64."""
    import oracle
    return oracle.to_f64(a, dt)


def rms(ref: np.ndarray) -> float:
    f = ref[np.isfinite(ref)]
    return float(np.sqrt(np.mean(f * f))) if f.size else 0.0


def assert_nan_match(got: np.ndarray, ref: np.ndarray, what: str):
    gn, rn = np.isnan(got), np.isnan(ref)
    if not np.array_equal(gn, rn):
        bad = np.argwhere(gn != rn)[:5]
        raise AssertionError(f"{what}: NaN positions differ at {bad.tolist()}")


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert_nan_match(got, ref, what)
    m = ~np.isnan(ref)
    if not m.any():
        return
    err = np.abs(got[m] - ref[m])
    r = rms(ref)
    if dtype == "f32":
        bound = 1e-4 * np.abs(ref[m]) + 1e-6 * r
        if not np.all(err <= bound):
            i = int(np.argmax(err - bound))
            raise AssertionError(
                f"{what}: FP32 element error {err[i]:.3e} > bound {bound[i]:.3e} "
                f"(ref {ref[m][i]:.6e}, got {got[m][i]:.6e})")
        mx = np.max(np.abs(ref[m]))
        assert err.max() <= 1e-4 * mx, f"{what}: FP32 max error {err.max():.3e} > 1e-4*max|ref|"
    else:
        bound = 2e-2 * r
        if err.max() > bound:
            i = int(np.argmax(err))
            raise AssertionError(
                f"{what}: {dtype} max abs error {err.max():.4e} > 2e-2*RMS = {bound:.4e} "
                f"(ref {ref[m][i]:.5e}, got {got[m][i]:.5e})")


def per_expert_sets(src_of: np.ndarray, offsets: np.ndarray):
    return [sorted(src_of[offsets[e]:offsets[e + 1]].tolist())
            for e in range(len(offsets) - 1)]


def np_of(t: torch.Tensor) -> np.ndarray:
    """Oracle-storage numpy copy of a tensor (raw words for 16-bit types)."""
    return W.to_numpy(t)
