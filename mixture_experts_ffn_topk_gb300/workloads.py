"""Seeded synthetic workloads for the local MoE FFN forward.

This module only draws random inputs; it holds none of the method's
arithmetic (no softmax, selection, dispatch, GEMM or norm). Both the CUDA path
(tests, bench) and the CPU oracle (tests) are fed from it.

Shapes, value distributions and structure follow the five workloads the
method is measured on:

* ``tiny_fp32``            T=64 H=128 I=256 E=8 top_k=2, renormalised, FP32,
  with two rows tied for the first rank, two rows tied across the selection
  boundary, one row holding NaN and one row of only -inf.
* ``fine_prefill_bf16``    T=4096 H=2048 I=1408 E=64 top_k=6, not
  renormalised; logits N(0,1) cast to BF16; near-uniform routing.
* ``coarse_prefill_bf16``  T=16384 H=4096 I=14336 E=8 top_k=2, renormalised;
  FP32 logits N(0,1) plus a per-expert bias N(0, 0.5) (mild imbalance).
* ``decode_bf16``          T=128 H=7168 I=2048 E=256 top_k=8, renormalised;
  FP32 logits N(0,1) plus a Zipf(s=1.1) per-expert bias, so many experts get
  no token and a few get many.
* ``combine_norm_bf16``    combine + residual Add + RMSNorm, T=8192 H=7168
  top_k=8 E=256: expert outputs [T*8, H] N(0,1) BF16, FP32 logits N(0,1) to
  route with, residual N(0,1) BF16, gamma N(1, 0.1) BF16, eps 1e-6.
* ``sigmoid_grouped_decode_bf16``  the decode shapes routed by group-limited
  sigmoid routing: 8 groups of 32 experts, 4 kept, each scored by its two
  best corrected scores, top_k=8, renormalised, scale 2.5; FP32 logits
  N(0,1) and an FP32 correction bias N(0, 0.01) drawn by its own generator.

N(m, v) names the variance v; expert weights are N(0, 1/fan_in). BF16 inputs
are FP32 draws rounded to nearest-even by torch's dtype cast. Seeds are
1000 + the workload's number (1..5) unless given.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class MoeConfig:
    name: str
    number: int
    T: int
    H: int
    I: int
    E: int
    top_k: int
    renormalize: bool
    dtype: str          # "f32" | "bf16" | "f16": x, weights, outputs
    logits_dtype: str   # "f32" | "bf16" | "f16"
    logit_bias: str = "none"   # "none" | "normal" | "zipf"
    bias_param: float = 0.0    # variance of the normal bias, or Zipf s
    special_rows: bool = False
    # routing: "softmax" (top-k of the softmax) or "sigmoid_grouped"
    # (group-limited sigmoid routing with the fields below)
    routing: str = "softmax"
    groups: int = 1
    selected_groups: int = 1
    group_top_two: bool = False
    scale: float = 1.0
    correction_var: float = 0.0   # variance of the FP32 correction bias (0: none)

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def assignments(self) -> int:
        return self.T * self.top_k

    def scaled(self, **kw) -> "MoeConfig":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class CombineNormConfig:
    name: str
    number: int
    T: int
    H: int
    E: int
    top_k: int
    eps: float
    dtype: str = "bf16"
    gamma_dtype: str = "bf16"

    @property
    def seed(self) -> int:
        return 1000 + self.number

    def scaled(self, **kw) -> "CombineNormConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny_fp32": MoeConfig("tiny_fp32", 1, T=64, H=128, I=256, E=8, top_k=2,
                           renormalize=True, dtype="f32", logits_dtype="f32",
                           special_rows=True),
    "fine_prefill_bf16": MoeConfig("fine_prefill_bf16", 2, T=4096, H=2048,
                                   I=1408, E=64, top_k=6, renormalize=False,
                                   dtype="bf16", logits_dtype="bf16"),
    "coarse_prefill_bf16": MoeConfig("coarse_prefill_bf16", 3, T=16384, H=4096,
                                     I=14336, E=8, top_k=2, renormalize=True,
                                     dtype="bf16", logits_dtype="f32",
                                     logit_bias="normal", bias_param=0.5),
    "decode_bf16": MoeConfig("decode_bf16", 4, T=128, H=7168, I=2048, E=256,
                             top_k=8, renormalize=True, dtype="bf16",
                             logits_dtype="f32", logit_bias="zipf",
                             bias_param=1.1),
    "sigmoid_grouped_decode_bf16": MoeConfig(
        "sigmoid_grouped_decode_bf16", 6, T=128, H=7168, I=2048, E=256, top_k=8,
        renormalize=True, dtype="bf16", logits_dtype="f32", routing="sigmoid_grouped",
        groups=8, selected_groups=4, group_top_two=True, scale=2.5, correction_var=0.01),
}

COMBINE_NORM = CombineNormConfig("combine_norm_bf16", 5, T=8192, H=7168, E=256,
                                 top_k=8, eps=1e-6)


@dataclasses.dataclass(frozen=True)
class CombineV2Config:
    """The Ascend V2 combine's extras on the combine + norm workload's shapes:
    special experts after the E routed ones, a shared expert, a 2-D active
    mask keeping each slot with probability keep."""
    name: str
    number: int
    T: int
    H: int
    E: int
    top_k: int
    eps: float
    zero: int
    copy: int
    const: int
    keep: float

    @property
    def seed(self) -> int:
        return 1000 + self.number


COMBINE_V2 = CombineV2Config("combine_v2_norm_bf16", 7, T=8192, H=7168, E=256, top_k=8,
                             eps=1e-6, zero=2, copy=2, const=4, keep=0.9)

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16,
                "f16": torch.float16}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, std=1.0, mean=0.0, dtype="f32", chunk_rows=None):
    """N(mean, std^2) drawn in FP32, then cast (RNE) to ``dtype``. Large
    tensors are drawn slab by slab along dim 0 to bound FP32 temporaries."""
    tdt = TORCH_DTYPES[dtype]
    out = torch.empty(shape, dtype=tdt, device=device)
    n0 = shape[0]
    step = chunk_rows or n0
    for s in range(0, n0, step):
        e = min(n0, s + step)
        v = torch.randn((e - s,) + tuple(shape[1:]), generator=g,
                        device=device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        if mean != 0.0:
            v.add_(mean)
        out[s:e].copy_(v)
    return out


def _logits(cfg: MoeConfig, g, device) -> torch.Tensor:
    l = torch.randn((cfg.T, cfg.E), generator=g, device=device,
                    dtype=torch.float32)
    if cfg.logit_bias == "normal":
        l += math.sqrt(cfg.bias_param) * torch.randn(
            (cfg.E,), generator=g, device=device, dtype=torch.float32)
    elif cfg.logit_bias == "zipf":
        # log of a Zipf(s) pmf up to a constant, over a seeded ranking
        rank = torch.randperm(cfg.E, generator=g, device=device) + 1
        l += -cfg.bias_param * torch.log(rank.to(torch.float32))
    if cfg.special_rows:
        _plant_special_rows(l, cfg.E)
    return l.to(TORCH_DTYPES[cfg.logits_dtype])


def _plant_special_rows(l: torch.Tensor, E: int) -> None:
    """Rows 0-1: two experts tie for the first rank; rows 2-3: two experts tie
    across the top_k=2 selection boundary; row 4 holds one NaN; row 5 is all
    -inf. Needs E >= 8 and T >= 6."""
    assert E >= 8 and l.shape[0] >= 6
    l[0, 2] = l[0, 6] = 5.0
    l[1, 1] = l[1, 4] = 5.0
    l[2, 7] = 5.0
    l[2, 3] = l[2, 5] = 4.0
    l[3, 0] = 5.0
    l[3, 2] = l[3, 6] = 4.0
    l[4, 3] = float("nan")
    l[5, :] = float("-inf")


def moe_inputs(cfg: MoeConfig, device="cpu", seed: int | None = None,
               weights_device=None) -> dict:
    """x [T,H], logits [T,E], gate/up [E,I,H], down [E,H,I] as torch tensors.

    Logits and x are always drawn by a CPU generator (so the routing of a
    workload is the same whatever device the tensors end up on) and moved to
    ``device``. The expert weights are drawn by a generator on
    ``weights_device`` (default ``device``), which lets multi-GB weights be
    drawn in place on a GPU. Same seed and devices -> same bytes."""
    seed = cfg.seed if seed is None else seed
    g = _gen(seed, "cpu")
    logits = _logits(cfg, g, "cpu").to(device)
    x = _normal((cfg.T, cfg.H), g, "cpu", dtype=cfg.dtype).to(device)
    wdev = device if weights_device is None else weights_device
    gw = _gen(seed + 7919, wdev)
    rows = max(1, (1 << 24) // max(1, cfg.I * cfg.H))
    gate = _normal((cfg.E, cfg.I, cfg.H), gw, wdev, std=cfg.H ** -0.5,
                   dtype=cfg.dtype, chunk_rows=rows)
    up = _normal((cfg.E, cfg.I, cfg.H), gw, wdev, std=cfg.H ** -0.5,
                 dtype=cfg.dtype, chunk_rows=rows)
    down = _normal((cfg.E, cfg.H, cfg.I), gw, wdev, std=cfg.I ** -0.5,
                   dtype=cfg.dtype, chunk_rows=rows)
    out = {"x": x, "logits": logits, "gate": gate, "up": up, "down": down}
    if cfg.routing == "sigmoid_grouped":
        b = correction_bias(cfg, device, seed)
        if b is not None:
            out["bias"] = b
    return out


def correction_bias(cfg: MoeConfig, device="cpu", seed: int | None = None):
    """FP32 [E] correction bias N(0, correction_var) for sigmoid routing, or
    None; drawn by a generator of its own (seed + 31) on the CPU."""
    if cfg.correction_var <= 0.0:
        return None
    seed = cfg.seed if seed is None else seed
    g = _gen(seed + 31, "cpu")
    b = torch.randn((cfg.E,), generator=g, dtype=torch.float32) * math.sqrt(cfg.correction_var)
    return b.to(device)


def combine_norm_inputs(cfg: CombineNormConfig, device="cpu",
                        seed: int | None = None) -> dict:
    """Expert outputs ``out_disp [T*top_k, H]``, routing logits ``[T, E]``
    (FP32, drawn on the CPU), ``residual [T, H]`` and ``gamma [H]`` (drawn on
    ``device``)."""
    seed = cfg.seed if seed is None else seed
    logits = torch.randn((cfg.T, cfg.E), generator=_gen(seed, "cpu"),
                         dtype=torch.float32).to(device)
    g = _gen(seed + 7919, device)
    rows = max(1, (1 << 24) // cfg.H)
    out_disp = _normal((cfg.T * cfg.top_k, cfg.H), g, device, dtype=cfg.dtype,
                       chunk_rows=rows)
    residual = _normal((cfg.T, cfg.H), g, device, dtype=cfg.dtype,
                       chunk_rows=rows)
    gamma = _normal((cfg.H,), g, device, std=math.sqrt(0.1), mean=1.0,
                    dtype=cfg.gamma_dtype)
    return {"out_disp": out_disp, "logits": logits, "residual": residual,
            "gamma": gamma}


def to_numpy(t: torch.Tensor):
    """Host numpy view in the oracle's storage convention (raw 16-bit words
    for bf16/f16)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_numpy(a, dtype: str, device="cpu") -> torch.Tensor:
    """Inverse of :func:`to_numpy`."""
    import numpy as np
    a = np.ascontiguousarray(a)
    if dtype in ("bf16", "f16"):
        t = torch.from_numpy(a.view(np.int16)).view(TORCH_DTYPES[dtype])
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def training_grad(cfg: MoeConfig, device="cpu", seed: int | None = None) -> torch.Tensor:
    """Upstream gradient of the MoE output for a training step: N(0, 1)
    ``[T, H]`` in the activation dtype, drawn by a CPU generator of its own
    (seed + 101) and moved to ``device``."""
    seed = cfg.seed if seed is None else seed
    g = _gen(seed + 101, "cpu")
    return _normal((cfg.T, cfg.H), g, "cpu", dtype=cfg.dtype).to(device)


def combine_v2_inputs(cfg: CombineV2Config, device="cpu", seed: int | None = None) -> dict:
    """Routing logits ``[T, E + special]`` FP32 and the 2-D mask (CPU
    generator), then on ``device``: expert outputs ``[T*top_k, H]``, ori_x,
    shared_x and residual ``[T, H]`` N(0,1), gamma N(1, 0.1), const alphas
    U(0, 2) / U(-1, 1) and const values N(0,1) ``[const, H]``, all BF16."""
    seed = cfg.seed if seed is None else seed
    special = cfg.zero + cfg.copy + cfg.const
    gc = _gen(seed, "cpu")
    logits = torch.randn((cfg.T, cfg.E + special), generator=gc, dtype=torch.float32)
    mask = torch.rand((cfg.T, cfg.top_k), generator=gc) < cfg.keep
    g = _gen(seed + 7919, device)
    rows = max(1, (1 << 24) // cfg.H)
    n = lambda shape: _normal(shape, g, device, dtype="bf16", chunk_rows=rows)
    out = {"logits": logits.to(device), "mask": mask.to(device),
           "out_disp": n((cfg.T * cfg.top_k, cfg.H)), "ori_x": n((cfg.T, cfg.H)),
           "shared_x": n((cfg.T, cfg.H)), "residual": n((cfg.T, cfg.H)),
           "gamma": _normal((cfg.H,), g, device, std=math.sqrt(0.1), mean=1.0, dtype="bf16"),
           "const_v": n((max(cfg.const, 1), cfg.H))}
    out["alpha1"] = (torch.rand((max(cfg.const, 1),), generator=g, device=device) * 2).to(torch.bfloat16)
    out["alpha2"] = (torch.rand((max(cfg.const, 1),), generator=g, device=device) * 2 - 1).to(torch.bfloat16)
    return out
