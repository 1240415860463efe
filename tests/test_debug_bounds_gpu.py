"""The bounds-checking build of the library (MOE_DEBUG_BOUNDS): the same C
ABI with device-side checks of the indices the kernels read from buffers,
standing in for a memory checker. Loaded here through its own handle, so
its status word is its own.

* On valid inputs it computes what the normal build computes (the one-call
  forward against the oracle, the dispatch bit for bit) and records nothing.
* Expert offsets that fall (a caller error moe_experts_forward cannot see on
  the host) are caught on the device: MOE_ERR_BOUNDS, nothing written. The
  case is chosen so that even the normal build stays inside every buffer
  (the falling expert has a negative row count, so no tiles).
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, to_f64

pytestmark = pytest.mark.gpu

BF16 = 1
BOUNDS = 10          # MOE_ERR_BOUNDS


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    path = build.build(debug_bounds=True)
    lib = moe.load_library(path)
    assert lib.moe_abi_version() == moe.load_library().moe_abi_version()
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_forward_clean_in_bounds_build(dbg):
    cfg = W.MoeConfig("dbg_fwd_bf16", 97, T=640, H=256, I=192, E=4, top_k=2, renormalize=True,
                      dtype="bf16", logits_dtype="f32", logit_bias="normal", bias_param=0.5)
    dev = torch.device("cuda:0")
    g = {n: v.to(dev) for n, v in W.moe_inputs(cfg, device="cpu").items()}
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    ws_n = dbg.moe_forward_workspace_size(T, H, I, E, k, BF16, 0)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    s = _stream()
    assert dbg.moe_device_status(s, 1) == 0
    rc = dbg.moe_forward(_p(g["x"]), BF16, _p(g["logits"]), 0, _p(g["gate"]), _p(g["up"]),
                         _p(g["down"]), T, H, I, E, k, 1, _p(y), _p(ws), ws_n, s)
    assert rc == 0, dbg.moe_last_error_detail()
    assert dbg.moe_device_status(s, 1) == 0
    o = {n: np_of(v.cpu()) for n, v in g.items()}
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"], o["up"],
                         o["down"], k, cfg.renormalize)
    assert_close(to_f64(y), ref["y"], cfg.dtype, "bounds-checking build y")


def test_dispatch_same_bits_in_bounds_build(dbg):
    dev = torch.device("cuda:0")
    T, k, E, H = 20000, 6, 64, 64
    gen = torch.Generator().manual_seed(5)
    idx = torch.randint(0, E, (T, k), generator=gen, dtype=torch.int32).to(dev)
    x = torch.randn((T, H), generator=gen).to(torch.bfloat16).to(dev)
    ref = moe.moe_dispatch(idx, x, E)
    out = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "row_of": torch.empty(T * k, dtype=torch.int32, device=dev),
           "src_of": torch.empty(T * k, dtype=torch.int32, device=dev),
           "x_disp": torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)}
    ws_n = dbg.moe_dispatch_workspace_size(T, k, E)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    s = _stream()
    rc = dbg.moe_dispatch(_p(idx), T, k, E, _p(x), BF16, H, _p(out["counts"]),
                          _p(out["offsets"]), _p(out["row_of"]), _p(out["src_of"]),
                          _p(out["x_disp"]), _p(ws), ws_n, s)
    assert rc == 0
    assert dbg.moe_device_status(s, 1) == 0
    for name in out:
        assert torch.equal(out[name], ref[name]), name


def test_falling_offsets_caught(dbg):
    dev = torch.device("cuda:0")
    E, H, I, rows = 3, 128, 64, 150
    gen = torch.Generator().manual_seed(6)
    x = torch.randn((rows, H), generator=gen).to(torch.bfloat16).to(dev)
    gate = (torch.randn((E, I, H), generator=gen) * H ** -0.5).to(torch.bfloat16).to(dev)
    up = (torch.randn((E, I, H), generator=gen) * H ** -0.5).to(torch.bfloat16).to(dev)
    down = (torch.randn((E, H, I), generator=gen) * I ** -0.5).to(torch.bfloat16).to(dev)
    offsets = torch.tensor([0, 100, 50, 150], dtype=torch.int32, device=dev)   # falls at expert 1
    out = torch.full((rows, H), 7.0, dtype=torch.float32, device=dev)
    ws_n = dbg.moe_experts_workspace_size(rows, E, H, I, BF16)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    s = _stream()
    assert dbg.moe_device_status(s, 1) == 0
    rc = dbg.moe_experts_forward(_p(x), _p(offsets), rows, _p(gate), _p(up), _p(down), E, H, I,
                                 BF16, _p(out), 0, _p(ws), ws_n, s)
    assert rc == 0
    assert dbg.moe_device_status(s, 1) == BOUNDS
    assert bool(torch.all(out == 7.0))          # nothing computed, nothing written
    assert dbg.moe_device_status(s, 1) == 0
