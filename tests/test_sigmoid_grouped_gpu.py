"""Group-limited sigmoid routing on the GPU against the CPU oracle (ruDNN user
guide, section 10, whose tie rule gives equal scores to the lower id), and
the one-call forward built on it.

Expert ids are compared bit-exactly on every row. Both sides round the
sigmoid once to FP32 from a double evaluation, so every decision (the kept
groups, the picked experts and their order) compares the same FP32 values,
including the equal group sums the small-integer inputs build on purpose
(sigmoid(x) + sigmoid(-x) = 1).
"""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_topk_gb300 as moe
import oracle
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def np_of(t):
    return W.to_numpy(t.cpu())


def to_f64(t):
    return t.detach().cpu().double().numpy()


def make_inputs(T, E, ldt, kind, with_bias, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "ties":
        l = torch.randint(-2, 3, (T, E), generator=g).float() * 0.5
    else:
        l = torch.randn((T, E), generator=g) * 1.5
    if kind == "specials":
        l[0, 3] = float("nan")
        l[1, :] = float("-inf")                  # valid: every score 0
        l[2, 5] = float("inf")                   # valid: score 1
        l[3, ::2] = float("inf")
        l[4, :] = 0.0                            # all tied
        l[5, :] = 30.0                           # all saturate to 1
    logits = l.to(W.TORCH_DTYPES[ldt])
    bias = None
    if with_bias:
        if kind == "ties":
            bias = (torch.randint(0, 2, (E,), generator=g).float() * 0.5).numpy().astype(np.float32)
        else:
            bias = (torch.randn((E,), generator=g) * 0.1).numpy().astype(np.float32)
    return logits, bias


# (T, E, groups, selected, top_k, top_two, renormalize, scale, logits dtype, kind, bias)
CASES = [
    (1000, 256, 8, 4, 8, True, True, 2.5, "f32", "normal", True),
    (600, 64, 8, 3, 6, False, False, 1.0, "bf16", "normal", False),
    (200, 1024, 128, 16, 64, True, True, 1.0, "f32", "normal", True),
    (300, 40, 1, 1, 5, False, True, 1.5, "f16", "normal", True),
    (257, 96, 3, 2, 7, True, False, 1.0, "bf16", "normal", True),
    (100, 7, 7, 7, 7, False, True, 1.0, "f32", "normal", False),
    (500, 32, 4, 2, 4, True, False, 1.0, "f32", "ties", True),
    (400, 48, 6, 2, 5, False, True, 1.0, "f32", "ties", False),
    (64, 24, 4, 2, 3, True, True, 2.0, "f32", "specials", True),
    (5000, 256, 8, 4, 8, True, True, 2.5, "bf16", "normal", True),
]


@pytest.mark.parametrize("T,E,G,S,k,two,ren,scale,ldt,kind,with_bias", CASES)
def test_route_sigmoid_grouped_parity(dev, T, E, G, S, k, two, ren, scale, ldt, kind, with_bias):
    logits, bias = make_inputs(T, E, ldt, kind, with_bias, seed=T * 7 + E)
    idx_ref, w_ref, _ = oracle.route_sigmoid_grouped(np_of(logits), ldt, bias, k, G, S, two,
                                                     ren, scale)
    bias_d = None if bias is None else torch.from_numpy(bias).to(dev)
    idx, w = moe.moe_route_sigmoid_grouped(logits.to(dev), bias_d, k, G, S, two, ren, scale)
    torch.cuda.synchronize()
    idx = idx.cpu().numpy().view(np.uint32)
    assert np.array_equal(idx, idx_ref), "expert ids differ"
    assert_close(to_f64(w), oracle.to_f64(w_ref, ldt), ldt, "weights")


def test_route_sigmoid_grouped_nan_bias_rows(dev):
    """A NaN correction makes every row's corrected scores hold a NaN."""
    T, E = 50, 16
    logits = torch.randn((T, E))
    bias = np.zeros(E, np.float32)
    bias[3] = np.nan
    idx, w = moe.moe_route_sigmoid_grouped(logits.to(dev), torch.from_numpy(bias).to(dev), 3,
                                           4, 2, True, True, 1.0)
    torch.cuda.synchronize()
    assert idx.cpu().tolist() == [[0, 1, 2]] * T
    assert torch.isnan(w.cpu()).all()


# ---------------------------------------------------------------- forward

FWD = [
    # (T, H, I, E, groups, selected, top_k, top_two, renormalize, scale, dtype)
    (300, 256, 128, 64, 8, 4, 6, True, True, 2.5, "bf16"),
    (2048, 256, 192, 16, 4, 2, 4, False, True, 1.0, "bf16"),     # >= 256 rows per expert: CTA pairs
    (200, 128, 64, 32, 4, 2, 3, True, False, 1.0, "f32"),
    (150, 192, 96, 24, 3, 3, 5, False, True, 1.5, "f16"),
]


@pytest.mark.parametrize("T,H,I,E,G,S,k,two,ren,scale,dt", FWD)
def test_forward_sigmoid_grouped_parity(dev, T, H, I, E, G, S, k, two, ren, scale, dt):
    cfg = W.MoeConfig("sg_fwd", 91, T=T, H=H, I=I, E=E, top_k=k, renormalize=ren, dtype=dt,
                      logits_dtype=dt)
    cpu = W.moe_inputs(cfg, device="cpu")
    g = torch.Generator().manual_seed(T + E)
    bias = (torch.randn((E,), generator=g) * 0.1).numpy().astype(np.float32)
    o = {n: np_of(v) for n, v in cpu.items()}
    ref = oracle.forward_sigmoid_grouped(o["x"], dt, o["logits"], dt, bias, o["gate"], o["up"],
                                         o["down"], k, G, S, two, ren, scale)
    gpu = {n: v.to(dev) for n, v in cpu.items()}
    y = moe.moe_forward_sigmoid_grouped(gpu["x"], gpu["logits"], torch.from_numpy(bias).to(dev),
                                        gpu["gate"], gpu["up"], gpu["down"], k, G, S, two, ren,
                                        scale)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert_close(to_f64(y), ref["y"], dt, "y")
