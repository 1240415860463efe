"""Combine with special experts, a shared expert and an active mask (the local
math of aclnnMoeDistributeCombineAddRmsNormV2), dispatch that leaves special
experts out, and the standalone RMSNorm (ruDNN user guide, section 7), on the
GPU against the CPU oracle."""

import numpy as np
import pytest
import torch

import mixture_experts_ffn_topk_gb300 as moe
import oracle
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, per_expert_sets, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def routed(T, k, E, special, seed):
    """Routing over E routed + `special` special experts (softmax top-k of the
    oracle), and the oracle's dispatch map of the routed ones."""
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn((T, E + special), generator=g).numpy().astype(np.float32)
    idx, w, _ = oracle.route(logits, "f32", k, True)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E)   # special ids: no row
    return idx, w, offsets, row_of, src_of


# (T, k, H, E, zero, copy, const, mask, shared, norm, expert-output dtype, dtype)
CASES = [
    (300, 4, 256, 8, 1, 1, 2, None, True, False, "f32", "bf16"),
    (300, 4, 256, 8, 1, 1, 2, "2d", True, True, "f32", "bf16"),
    (257, 6, 512, 16, 2, 0, 0, "1d", False, True, "bf16", "bf16"),
    (128, 2, 128, 4, 0, 2, 0, "2d", False, False, "f16", "f16"),
    (200, 3, 192, 6, 0, 0, 3, None, True, True, "f32", "f32"),
    (129, 8, 7168, 32, 2, 2, 2, "2d", True, True, "f32", "bf16"),
    (64, 2, 64, 4, 0, 0, 0, "1d", True, False, "f32", "bf16"),
]


@pytest.mark.parametrize("T,k,H,E,zero,copy,const,mask,shared,norm,odt,dt", CASES)
def test_combine_v2_parity(dev, T, k, H, E, zero, copy, const, mask, shared, norm, odt, dt):
    special = zero + copy + const
    idx, w, offsets, row_of, _ = routed(T, k, E, special, seed=T + H)
    rows = int(offsets[E])
    g = torch.Generator().manual_seed(H)
    tdt = W.TORCH_DTYPES[dt]
    out_disp = torch.randn((max(rows, 1), H), generator=g).to(W.TORCH_DTYPES[odt])
    ori_x = torch.randn((T, H), generator=g).to(tdt) if (copy or const) else None
    a1 = (torch.rand((const,), generator=g) * 2).to(tdt) if const else None
    a2 = (torch.rand((const,), generator=g) * 2 - 1).to(tdt) if const else None
    cv = torch.randn((const, H), generator=g).to(tdt) if const else None
    shx = torch.randn((T, H), generator=g).to(tdt) if shared else None
    m = None
    if mask == "1d":
        m = torch.arange(T) < (T * 7) // 10          # kept tokens first
    elif mask == "2d":
        m = torch.rand((T, k), generator=g) < 0.7
    residual = torch.randn((T, H), generator=g).to(tdt) if norm else None
    gamma = (1 + 0.1 * torch.randn((H,), generator=g)).to(torch.float32) if norm else None

    on = lambda t: None if t is None else t.to(dev)
    o = lambda t: None if t is None else np_of(t)
    ref = oracle.combine_v2(np_of(out_disp), odt, w, "f32", row_of, k, dt, ids=idx, E=E,
                            zero=zero, copy=copy, const=const, ori_x=o(ori_x), alpha1=o(a1),
                            alpha2=o(a2), const_v=o(cv), shared_x=o(shx),
                            mask=None if m is None else m.numpy())
    res = moe.moe_combine_v2(on(out_disp), torch.from_numpy(w).to(dev),
                             torch.from_numpy(row_of).to(dev), tdt,
                             expert_indices=torch.from_numpy(idx.view(np.int32)).to(dev),
                             num_experts=E, zero_experts=zero, copy_experts=copy,
                             const_experts=const, ori_x=on(ori_x), const_alpha1=on(a1),
                             const_alpha2=on(a2), const_v=on(cv), shared_expert_x=on(shx),
                             active_mask=on(m), residual=on(residual), gamma=on(gamma),
                             eps=1e-6)
    torch.cuda.synchronize()
    if not norm:
        assert_close(to_f64(res), ref, dt, "combineOut")
        return
    y, x_out, rstd = res
    y_ref, x_ref, r_ref = oracle.add_rmsnorm(ref, np_of(residual), dt, np_of(gamma), "f32", 1e-6)
    assert_close(to_f64(x_out), oracle.to_f64(x_ref, dt), dt, "x_out")
    assert_close(to_f64(y), oracle.to_f64(y_ref, dt), dt, "y")
    assert_close(rstd.cpu().numpy().astype(np.float64), r_ref.astype(np.float64), "f32", "rstd")


def test_combine_v2_nan_rows(dev):
    """An id past the last special expert, or a routed slot without a row,
    makes the token's row NaN; other rows are untouched by it."""
    T, k, H, E = 6, 2, 64, 4
    idx = np.array([[0, 1], [1, 7], [2, 4], [3, 5], [0, 9], [1, 2]], np.uint32)
    row_of = np.array([0, 1, 2, -1, 3, -1, 4, -1, 5, -1, 6, 7], np.int32)
    row_of[4] = -1                                   # token 2 slot 0: routed id 2, no row
    w = np.full((T, k), 0.5, np.float32)
    out = torch.randn((8, H)).float()
    ori = torch.randn((T, H)).bfloat16()
    ref = oracle.combine_v2(np_of(out), "f32", w, "f32", row_of, k, "bf16", ids=idx, E=E,
                            zero=1, copy=1, ori_x=np_of(ori))
    y = moe.moe_combine_v2(out.to(dev), torch.from_numpy(w).to(dev),
                           torch.from_numpy(row_of).to(dev), torch.bfloat16,
                           expert_indices=torch.from_numpy(idx.view(np.int32)).to(dev),
                           num_experts=E, zero_experts=1, copy_experts=1, ori_x=ori.to(dev))
    torch.cuda.synchronize()
    nan_ref = np.isnan(ref).all(axis=1)
    assert nan_ref.tolist() == [False, True, True, False, True, False]
    assert_close(to_f64(y), ref, "bf16", "combineOut with NaN rows")


def test_dispatch_special(dev):
    """Special ids get no row and raise no bad-index status; an id past them
    still does."""
    T, k, E, special, H = 500, 4, 16, 3, 64
    idx, _, offsets, row_of, src_of = routed(T, k, E, special, seed=5)
    assert (idx >= E).any()
    x = torch.randn((T, H)).bfloat16().to(dev)
    moe.moe_device_status(clear=True)
    d = moe.moe_dispatch_special(torch.from_numpy(idx.view(np.int32)).to(dev), x, E, special)
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=True) == 0
    assert np.array_equal(d["offsets"].cpu().numpy(), offsets)
    g_row = d["row_of"].cpu().numpy()
    assert np.array_equal(g_row < 0, row_of < 0)
    g_src = d["src_of"].cpu().numpy()
    assert per_expert_sets(g_src, offsets) == per_expert_sets(src_of, offsets)
    bad = idx.copy()
    bad[7, 1] = E + special
    moe.moe_dispatch_special(torch.from_numpy(bad.view(np.int32)).to(dev), x, E, special)
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=True) != 0


# (rows, H, dtype, gamma dtype)
NORM_CASES = [(1000, 2048, "bf16", "f32"), (77, 264, "f16", "f16"), (300, 7168, "bf16", "bf16"),
              (64, 128, "f32", "f32"), (5, 16384, "bf16", "f32"), (0, 64, "bf16", "f32")]


@pytest.mark.parametrize("rows,H,dt,gdt", NORM_CASES)
def test_rmsnorm_parity(dev, rows, H, dt, gdt):
    g = torch.Generator().manual_seed(rows + H)
    x = (torch.randn((rows, H), generator=g) * 3).to(W.TORCH_DTYPES[dt])
    gamma = (1 + 0.1 * torch.randn((H,), generator=g)).to(W.TORCH_DTYPES[gdt])
    y, rstd = moe.moe_rmsnorm(x.to(dev), gamma.to(dev), 1e-6)
    torch.cuda.synchronize()
    if rows == 0:
        return
    y_ref, r_ref = oracle.rmsnorm(np_of(x), dt, np_of(gamma), gdt, 1e-6)
    assert_close(to_f64(y), oracle.to_f64(y_ref, dt), dt, "y")
    assert_close(rstd.cpu().numpy().astype(np.float64), r_ref.astype(np.float64), "f32", "rstd")
