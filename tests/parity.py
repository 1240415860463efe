"""Tolerances and helpers for comparing the CUDA path with the CPU oracle.

Bars (fixed once here, used by every parity test):

* integer and index outputs (expert ids, counts, offsets, dispatch maps,
  gathered rows): bit-exact; dispatch rows are compared as a per-expert set
  because the order inside an expert is left open by the pages;
* FP32 outputs, "within 1e-4 relative error": the largest error is at most
  ``1e-4 * max|ref|`` (max-norm relative error of the tensor), and every
  element is within ``1e-4 * |ref| + 1e-5 * RMS(ref)``; the RMS floor admits
  the FP32 cancellation error of elements whose value is far below the
  tensor's scale (a length-K FP32 dot product carries about sqrt(K) * 2^-24
  of its terms' magnitude);
* BF16 / F16 outputs, "max abs error <= 2e-2 x output RMS against an FP32
  oracle fed the same rounded inputs": for every element,
  ``|got - ref| - ulp(ref)/2 <= 2e-2 * RMS(ref)``, where ``ulp(ref)/2`` is half
  the spacing of the output dtype at ``ref`` -- the error that rounding the
  exact value once to the output dtype makes by itself. Without that term a
  correctly rounded exact result already fails on outputs whose max|y|/RMS
  exceeds ~10 (bf16 half-ulp is 2^-9 |y|), which the routed MoE outputs reach;
* NaN positions must match exactly in every case; RMS is taken over the
  finite reference entries;
* training backward: the bar above covers products with ONE operand that this
  design rounds to BF16/F16 on its way (the forward's h). In the chained
  backward, every tensor-core product has two such operands (the output
  gradient rounded to the activation dtype by the combine backward, times h,
  dg or du, themselves rounded), and independent roundings add, so those
  results take ``rounds=2``: ``2 * 2e-2 * RMS``. An emulation of exactly these
  roundings on the test shapes reaches 0.028 x RMS (one rounding: 0.018).
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


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, rounds: int = 1):
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
        bound = 1e-4 * np.abs(ref[m]) + 1e-5 * r
        if not np.all(err <= bound):
            i = int(np.argmax(err - bound))
            raise AssertionError(
                f"{what}: FP32 element error {err[i]:.3e} > bound {bound[i]:.3e} "
                f"(ref {ref[m][i]:.6e}, got {got[m][i]:.6e})")
        mx = np.max(np.abs(ref[m]))
        assert err.max() <= 1e-4 * mx, f"{what}: FP32 max error {err.max():.3e} > 1e-4*max|ref|"
    else:
        half_ulp = half_ulp_of(ref[m], dtype)
        excess = err - half_ulp
        bound = 2e-2 * rounds * r
        if excess.max() > bound:
            i = int(np.argmax(excess))
            raise AssertionError(
                f"{what}: {dtype} error {err[i]:.4e} - half ulp {half_ulp[i]:.3e} > "
                f"{2e-2 * rounds:g}*RMS = {bound:.4e} (ref {ref[m][i]:.5e}, got {got[m][i]:.5e})")


def half_ulp_of(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half the spacing of ``dtype`` at |ref| (the bound on one correct
    round-to-nearest): bf16 keeps 8 significant bits, f16 11 (with its
    subnormal spacing 2^-24 as the floor)."""
    a = np.abs(ref)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    if dtype == "bf16":
        e = np.maximum(e, -126)
        return np.exp2(e - 8)
    if dtype == "f16":
        e = np.maximum(e, -14)
        return np.exp2(e - 11)
    raise ValueError(dtype)


def per_expert_sets(src_of: np.ndarray, offsets: np.ndarray):
    return [sorted(src_of[offsets[e]:offsets[e + 1]].tolist())
            for e in range(len(offsets) - 1)]


def np_of(t: torch.Tensor) -> np.ndarray:
    """Oracle-storage numpy copy of a tensor (raw words for 16-bit types)."""
    return W.to_numpy(t)
