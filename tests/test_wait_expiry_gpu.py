"""The bounded device waits' failure path, run on the GPU without a fault
(the error convention of the ruDNN user guide, section 3: a status, not a
hang).

moe_selftest_wait_expiry launches the folded second expert GEMM of the
one-call forward on its own, with per-expert readiness counters that no
first GEMM ever raises. With the wait limit shortened to a few milliseconds,
every producer gives up, the kernel records MOE_ERR_DEVICE_TIMEOUT, drains
and exits without writing its output; the device stays usable and the next
forward is correct.
"""

from __future__ import annotations

import time

import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, to_f64

pytestmark = pytest.mark.gpu

TIMEOUT = 8        # MOE_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


# (experts, rows per expert): CTA pairs (>= 256 rows per expert on average)
# and single CTAs
@pytest.mark.parametrize("E,rows_per_expert", [(2, 300), (4, 64)], ids=["pairs", "single"])
def test_unsatisfiable_wait_ends_in_timeout_status(dev, E, rows_per_expert):
    H, I = 256, 128
    assert moe.moe_device_status(clear=True) == 0
    y_acc = torch.zeros((E * rows_per_expert, H), dtype=torch.float32, device=dev)
    moe.moe_set_wait_limit_ns(2_000_000)                   # 2 ms
    try:
        assert moe.moe_wait_limit_ns() == 2_000_000
        t0 = time.perf_counter()
        moe.moe_selftest_wait_expiry(E, rows_per_expert, H, I, y_acc)
        status = moe.moe_device_status(clear=True)
        elapsed = time.perf_counter() - t0
    finally:
        moe.moe_set_wait_limit_ns(0)
    assert moe.moe_wait_limit_ns() == 2_000_000_000
    assert status == TIMEOUT
    assert elapsed < 5.0                                   # the short limit, not the default
    assert int(torch.count_nonzero(y_acc)) == 0            # nothing was reduced into y_acc
    # the status word was cleared, and the context still runs kernels
    assert moe.moe_device_status(clear=True) == 0


def test_forward_after_expiry_is_correct(dev):
    moe.moe_set_wait_limit_ns(2_000_000)
    try:
        y_acc = torch.zeros((600, 256), dtype=torch.float32, device=dev)
        moe.moe_selftest_wait_expiry(2, 300, 256, 128, y_acc)
        assert moe.moe_device_status(clear=True) == TIMEOUT
    finally:
        moe.moe_set_wait_limit_ns(0)
    cfg = W.MoeConfig("after_expiry_bf16", 96, T=700, H=256, I=192, E=2, top_k=1,
                      renormalize=True, dtype="bf16", logits_dtype="bf16")
    g = {n: v.to(dev) for n, v in W.moe_inputs(cfg, device="cpu").items()}
    y = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                        cfg.renormalize)
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=True) == 0
    o = {n: np_of(v.cpu()) for n, v in g.items()}
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"], o["up"],
                         o["down"], cfg.top_k, cfg.renormalize)
    assert_close(to_f64(y), ref["y"], cfg.dtype, "y after a timed-out kernel")
