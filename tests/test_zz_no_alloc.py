"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device scratch (their device memory belongs to a pool that permits
no allocation after start-up, or they cannot afford the synchronisation
cudaMalloc brings on a latency-critical path). It keeps its scratch in a
256 KiB array the library owns on each device.

Checked through the C ABI (ctypes, raw pointers) against moe_dispatch with a
caller workspace, on two calls in a row with different inputs, so the second
call also shows that nothing left in the shared array from the first one
leaks into its result. Integer and copy outputs must be bit-exact, as in the
other dispatch tests. This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_ffn_topk_gb300 as moe

pytestmark = pytest.mark.gpu

BF16, F32 = 1, 0


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    return moe.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(T, k, E, H, dtype, dev):
    A = T * k
    return {"counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
            "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            "row_of": torch.full((A,), -7, dtype=torch.int32, device=dev),
            "src_of": torch.full((A,), -7, dtype=torch.int32, device=dev),
            "x_disp": torch.zeros((A, H), dtype=dtype, device=dev)}


def _case(lib, T, k, E, H, seed, dev):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int().to(dev)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16).to(dev)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ref = _outputs(T, k, E, H, x.dtype, dev)
    ws = torch.empty(lib.moe_dispatch_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    rc = lib.moe_dispatch(_p(idx), T, k, E, _p(x), BF16, H, _p(ref["counts"]),
                          _p(ref["offsets"]), _p(ref["row_of"]), _p(ref["src_of"]),
                          _p(ref["x_disp"]), _p(ws), ws.numel(), s)
    assert rc == 0

    got = _outputs(T, k, E, H, x.dtype, dev)
    rc = lib.moe_dispatch_noalloc(_p(idx), T, k, E, _p(x), BF16, H, _p(got["counts"]),
                                  _p(got["offsets"]), _p(got["row_of"]), _p(got["src_of"]),
                                  _p(got["x_disp"]), s)
    assert rc == 0, lib.moe_last_error_detail()
    torch.cuda.synchronize()
    assert lib.moe_device_status(s, 1) == 0
    for name in ("counts", "offsets", "row_of", "src_of", "x_disp"):
        assert torch.equal(got[name], ref[name]), name
    # and the result is a valid dispatch: every assignment has its own row
    row_of = got["row_of"].cpu().numpy()
    assert sorted(row_of.tolist()) == list(range(T * k))


def test_noalloc_matches_dispatch_on_two_calls(lib):
    dev = torch.device("cuda:0")
    # first call: many chunks, many experts (fills a large part of the array)
    _case(lib, T=8192, k=8, E=256, H=64, seed=1, dev=dev)
    # second call: different shape, fewer experts, reusing the same array
    _case(lib, T=4096, k=6, E=64, H=2048, seed=2, dev=dev)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    dev = torch.device("cuda:0")
    T, k, E, H = 32768, 8, 1024, 8
    # the dispatch workspace of this shape (per-chunk counts of 1024 experts,
    # about 4 MiB on a 152-SM GPU) is far beyond the 256 KiB array
    assert lib.moe_dispatch_workspace_size(T, k, E) > 256 * 1024
    idx = torch.zeros((T, k), dtype=torch.int32, device=dev)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    out = _outputs(T, k, E, H, x.dtype, dev)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.moe_dispatch_noalloc(_p(idx), T, k, E, _p(x), BF16, H, _p(out["counts"]),
                                  _p(out["offsets"]), _p(out["row_of"]), _p(out["src_of"]),
                                  _p(out["x_disp"]), s)
    assert rc == 6                       # MOE_ERR_WORKSPACE
    assert b"256 KiB" in lib.moe_last_error_detail()
    # a bad argument is reported as moe_dispatch would report it, before the
    # size test
    rc = lib.moe_dispatch_noalloc(_p(idx), T, k, E, _p(x), 7, H, _p(out["counts"]),
                                  _p(out["offsets"]), _p(out["row_of"]), _p(out["src_of"]),
                                  _p(out["x_disp"]), s)
    assert rc == 3                       # MOE_ERR_DTYPE
    torch.cuda.synchronize()
    assert torch.all(out["counts"] == -7)   # nothing was enqueued
