"""First-order MoE training (ruDNN user guide, section 12) on the GPU,
through the C ABI, against the CPU oracle on the same seeded bytes.

Covers the router weights of a fixed selection and their logits gradient
(softmax and sigmoid scoring, renormalisation, scale, repeated ids, illegal
ids, invalid rows, E up to 1024 and top_k up to 64, every logits and index
dtype), the combine and dispatch backward, the training forward's cache, the
expert backward (FP32 on CUDA cores, BF16/F16 on tcgen05: several 128-row
tiles, ragged K/N/M edges, experts without rows, segment tails in the weight
gradients) and the whole backward chain in the section's order.

Bars (``parity.py``): FP32 results within 1e-4 relative; results of a BF16 /
F16 computation within half an output ulp plus 2e-2 x RMS, including the
FP32 weight gradients of the BF16 expert backward (h and the dg / du
intermediates are BF16); 4e-2 x RMS where a product carries two roundings
of this design (the chained backward); NaN positions exact.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import TORCH_TO_NAME, assert_close, np_of, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


# ---------------------------------------------------------------- router

ROUTER_CASES = [
    # (T, E, k, logits dtype, index dtype, scoring, renorm, scale)
    (500, 64, 6, torch.bfloat16, torch.int32, "softmax", False, 1.0),
    (500, 64, 6, torch.float32, torch.int64, "softmax", True, 1.0),
    (300, 256, 8, torch.float32, torch.int32, "sigmoid", True, 2.5),
    (300, 256, 8, torch.bfloat16, torch.int64, "sigmoid", False, 1.0),
    (200, 1024, 64, torch.float32, torch.int32, "softmax", True, 1.5),
    (200, 1024, 40, torch.float16, torch.int32, "sigmoid", True, 1.0),
    (257, 7, 7, torch.float32, torch.int64, "softmax", False, 3.0),
    (64, 1, 1, torch.float32, torch.int32, "softmax", True, 1.0),
    (33, 48, 33, torch.float16, torch.int64, "softmax", True, 1.0),
]


def _router_inputs(T, E, k, ldt, idt, seed):
    g = _gen(seed)
    logits = (torch.randn((T, E), generator=g) * 1.5).to(ldt)
    # the selection: the routing's own top-k for most rows; repeated ids,
    # illegal ids and invalid softmax rows in a few
    idx = torch.topk(logits.float(), k, dim=1).indices
    if T > 8 and E > 1:
        idx[1, :] = idx[1, 0]                    # every slot the same expert
        idx[2, k - 1] = E                        # illegal: too large
        if idt != torch.uint32:
            idx[3, 0] = -1                       # illegal: negative
        logits[4, E // 2] = float("nan")
        logits[5, :] = float("-inf")
        logits[6, 0] = float("inf")
        logits[7, : E - 1] = float("-inf")       # a valid row with one finite logit
    gw = torch.randn((T, k), generator=g)
    return logits, idx.to(idt), gw


@pytest.mark.parametrize("case", ROUTER_CASES, ids=lambda c: f"T{c[0]}E{c[1]}k{c[2]}"
                         f"-{str(c[3])[6:]}-{c[5]}{'-renorm' if c[6] else ''}")
def test_router_weights_and_backward(dev, case):
    T, E, k, ldt, idt, scoring, renorm, scale = case
    logits, idx, gw = _router_inputs(T, E, k, ldt, idt, 7000 + T + E + k)
    name = TORCH_TO_NAME[ldt]
    w = moe.moe_router_weights(logits.to(dev), idx.to(dev), scoring, renorm, scale)
    dl = moe.moe_router_backward(logits.to(dev), idx.to(dev), gw.to(dev), scoring, renorm, scale)
    torch.cuda.synchronize()
    ref_w, _ = oracle.router_weights(np_of(logits), name, idx.numpy(), scoring, renorm, scale, "f64")
    ref_dl, _ = oracle.router_backward(np_of(logits), name, idx.numpy(), gw.numpy(), "f32",
                                       scoring, renorm, scale, "f64")
    assert_close(to_f64(w), ref_w, "f32", "router weights")
    assert_close(to_f64(dl), ref_dl, name, "router logits gradient")
    moe.moe_device_status(clear=True)


def test_router_unsigned_ids(dev):
    if not hasattr(torch, "uint32"):
        pytest.skip("torch has no uint32")
    T, E, k = 40, 16, 4
    logits, idx, gw = _router_inputs(T, E, k, torch.float32, torch.int64, 7100)
    ids = idx.numpy().astype(np.int64)
    ids[3, 0] = 0xFFFFFFFF                       # the u32 bit pattern of -1: an illegal id
    bits = torch.from_numpy(ids.astype(np.uint32).view(np.int32)).to(dev)
    try:
        u = bits.view(torch.uint32)
    except (RuntimeError, TypeError):
        pytest.skip("this torch cannot view int32 as uint32")
    w = moe.moe_router_weights(logits.to(dev), u, "softmax", True, 1.0)
    torch.cuda.synchronize()
    ref_w, _ = oracle.router_weights(logits.numpy(), "f32", ids.astype(np.uint32), "softmax",
                                     True, 1.0, "f64")
    assert_close(to_f64(w), ref_w, "f32", "router weights (u32 ids)")
    moe.moe_device_status(clear=True)


def test_router_bad_id_sets_status(dev):
    logits = torch.randn((16, 8), device=dev)
    idx = torch.zeros((16, 2), dtype=torch.int32, device=dev)
    idx[3, 1] = 8
    moe.moe_device_status(clear=True)
    w = moe.moe_router_weights(logits, idx)
    assert moe.moe_device_status(clear=True) == 9          # MOE_ERR_BAD_INDEX
    wn = w.cpu().numpy()
    assert np.isnan(wn[3]).all() and np.isfinite(np.delete(wn, 3, axis=0)).all()


def test_router_argument_errors(dev):
    logits = torch.randn((4, 8), device=dev)
    idx = torch.zeros((4, 2), dtype=torch.int32, device=dev)
    for kw in (dict(scale=0.0), dict(scale=float("inf"))):
        with pytest.raises(moe.MoeError) as e:
            moe.moe_router_weights(logits, idx, **kw)
        assert e.value.name == "MOE_ERR_VALUE"
    with pytest.raises(moe.MoeError) as e:
        moe.moe_router_weights(torch.randn((4, 80), device=dev),
                               torch.zeros((4, 65), dtype=torch.int32, device=dev))
    assert e.value.name == "MOE_ERR_SHAPE"


# ----------------------------------------------------- combine / dispatch backward

def _routed(T, E, k, seed):
    g = _gen(seed)
    logits = torch.randn((T, E), generator=g)
    idx, _, _ = oracle.route(logits.numpy(), "f32", k, True)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E)
    return idx, offsets, row_of, src_of


@pytest.mark.parametrize("dt,odt,wdt", [
    (torch.bfloat16, torch.float32, torch.float32),
    (torch.bfloat16, torch.bfloat16, torch.bfloat16),
    (torch.float16, torch.float16, torch.float32),
    (torch.float32, torch.float32, torch.float32),
])
def test_combine_backward(dev, dt, odt, wdt):
    T, E, k, H = 333, 16, 4, 264
    idx, offsets, row_of, src_of = _routed(T, E, k, 7200)
    g = _gen(7201)
    out = torch.randn((T * k, H), generator=g).to(odt)
    w = torch.rand((T, k), generator=g).to(wdt)
    gy = torch.randn((T, H), generator=g).to(dt)
    ro = row_of.copy()
    ro[5] = -1                                  # a slot without a row
    dexp, dw = moe.moe_combine_backward(out.to(dev), w.to(dev), torch.from_numpy(ro).to(dev),
                                        gy.to(dev))
    torch.cuda.synchronize()
    ref_dexp, ref_dw = oracle.combine_backward(np_of(out), TORCH_TO_NAME[odt], np_of(w),
                                               TORCH_TO_NAME[wdt], ro, np_of(gy),
                                               TORCH_TO_NAME[dt], k)
    named = ro[ro >= 0]
    assert_close(to_f64(dexp)[named], ref_dexp[named], TORCH_TO_NAME[dt], "expert-output gradient")
    assert_close(to_f64(dw), ref_dw, "f32", "routing-weight gradient")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("k", [1, 6, 40])
def test_dispatch_backward(dev, dt, k):
    T, E, H = 211, 48, 136
    idx, offsets, row_of, src_of = _routed(T, E, k, 7300 + k)
    d = torch.randn((T * k, H), generator=_gen(7301)).to(dt)
    ro = row_of.copy()
    ro[7] = -1
    dx = moe.moe_dispatch_backward(d.to(dev), torch.from_numpy(ro).to(dev), T, k)
    torch.cuda.synchronize()
    ref = oracle.dispatch_backward(np_of(d), TORCH_TO_NAME[dt], ro, k)
    assert_close(to_f64(dx), ref, TORCH_TO_NAME[dt], "dispatch backward")


# ---------------------------------------------------------------- experts

EXPERT_CASES = [
    # (name, T, H, I, E, k, dtype, zipf bias)
    ("ragged_bf16", 300, 320, 200, 6, 2, torch.bfloat16, 0.0),
    ("many_experts_bf16", 256, 256, 136, 64, 6, torch.bfloat16, 0.0),
    ("hot_expert_bf16", 400, 128, 264, 8, 2, torch.bfloat16, 3.0),
    ("single_expert_f16", 150, 192, 128, 1, 1, torch.float16, 0.0),
    ("ragged_f32", 200, 192, 136, 5, 2, torch.float32, 0.0),
    ("empty_experts_f16", 40, 256, 512, 32, 2, torch.float16, 2.0),
    # at least 2 x 128 rows per expert: dh and dx run on CTA pairs too; skewed
    # counts leave a pair's second M-tile past an expert's rows; H = I = 200
    # leave K and N tails
    ("pair_skewed_bf16", 900, 200, 200, 3, 1, torch.bfloat16, 1.0),
    ("pair_f16", 640, 384, 320, 4, 2, torch.float16, 0.0),
    # at least 2048 rows per expert on average: the backward GEMMs run on CTA
    # pairs as well (M = 256; weight gradients reduce over thousands of rows);
    # K / N / M tails, one expert, and a skewed split where one expert holds
    # few rows
    ("bwd_pairs_bf16", 4500, 200, 328, 2, 1, torch.bfloat16, 0.8),
    ("bwd_pairs_one_expert_f16", 5200, 264, 136, 1, 1, torch.float16, 0.0),
    ("bwd_pairs_skewed_bf16", 6400, 136, 200, 3, 1, torch.bfloat16, 3.0),
    # two experts without rows (their weight gradients written as zeros) and
    # one of 13 rows beside one of 8987
    ("bwd_pairs_empty_experts_bf16", 9000, 136, 200, 4, 1, torch.bfloat16, 6.0),
]


def _expert_inputs(case, dev):
    name, T, H, I, E, k, dt, zipf = case
    cfg = W.MoeConfig(name, 95, T=T, H=H, I=I, E=E, top_k=k, renormalize=True,
                      dtype=TORCH_TO_NAME[dt], logits_dtype="f32",
                      logit_bias="zipf" if zipf else "none", bias_param=zipf)
    cpu = W.moe_inputs(cfg, device="cpu")
    idx, _, _ = oracle.route(np_of(cpu["logits"]), "f32", k, True)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E)
    x_disp = torch.from_numpy(oracle.gather(np_of(cpu["x"]), TORCH_TO_NAME[dt], k, src_of, T * k))
    if dt != torch.float32:
        x_disp = x_disp.view(torch.int16).view(dt)
    dout = torch.randn((T * k, H), generator=_gen(7400 + T)).to(dt)
    on = {kk: cpu[kk].to(dev) for kk in ("gate", "up", "down")}
    return cfg, cpu, offsets, x_disp, dout, on


@pytest.mark.parametrize("case", EXPERT_CASES, ids=lambda c: c[0])
def test_experts_training_forward(dev, case):
    cfg, cpu, offsets, x_disp, dout, on = _expert_inputs(case, dev)
    dt = x_disp.dtype
    name = TORCH_TO_NAME[dt]
    off = torch.from_numpy(offsets).to(dev)
    xd = x_disp.to(dev)
    out_t, cache = moe.moe_experts_forward_training(xd, off, on["gate"], on["up"], on["down"],
                                                    out_dtype=torch.float32)
    out_f = moe.moe_experts_forward(xd, off, on["gate"], on["up"], on["down"],
                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    # the training forward computes exactly what the forward computes
    assert torch.equal(out_t, out_f)
    # cache: h [rows, I] in the expert dtype, then g and u [rows, I] in FP32
    rows, I = x_disp.shape[0], cfg.I
    hb = rows * I * x_disp.element_size()
    h_c = cache[:hb].view(dt).view(rows, I)
    gu_c = cache[hb: hb + 2 * rows * I * 4].view(torch.float32).view(2, rows, I)
    g, u, h = oracle.experts_cache_dispatched(np_of(x_disp), name, offsets, np_of(cpu["gate"]),
                                              np_of(cpu["up"]))
    # g and u are FP32 results of a computation in the expert dtype
    assert_close(to_f64(gu_c[0]), g, name, "cached g")
    assert_close(to_f64(gu_c[1]), u, name, "cached u")
    assert_close(to_f64(h_c), h, name, "cached h")


@pytest.mark.parametrize("case", EXPERT_CASES, ids=lambda c: c[0])
def test_experts_backward(dev, case):
    cfg, cpu, offsets, x_disp, dout, on = _expert_inputs(case, dev)
    dt = x_disp.dtype
    name = TORCH_TO_NAME[dt]
    off = torch.from_numpy(offsets).to(dev)
    xd = x_disp.to(dev)
    _, cache = moe.moe_experts_forward_training(xd, off, on["gate"], on["up"], on["down"])
    E, I, H = cfg.E, cfg.I, cfg.H
    nan = float("nan")
    gg = torch.full((E, I, H), nan, device=dev)
    gu = torch.full((E, I, H), nan, device=dev)
    gd = torch.full((E, H, I), nan, device=dev)
    dx, gg, gu, gd = moe.moe_experts_backward(xd, off, on["gate"], on["up"], on["down"], cache,
                                              dout.to(dev), grad_gate=gg, grad_up=gu,
                                              grad_down=gd)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.experts_backward_dispatched(np_of(x_disp), name, offsets, np_of(cpu["gate"]),
                                             np_of(cpu["up"]), np_of(cpu["down"]), np_of(dout),
                                             name)
    bar = name   # weight gradients of a BF16/F16 computation take its bar
    assert_close(to_f64(dx), ref[0], name, "grad x_disp")
    assert_close(to_f64(gg), ref[1], bar, "grad gate")
    assert_close(to_f64(gu), ref[2], bar, "grad up")
    assert_close(to_f64(gd), ref[3], bar, "grad down")


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_experts_backward_no_rows(dev, dt):
    """rows = 0: every weight gradient is written, as zeros."""
    E, H, I = 3, 64, 32
    g = torch.randn((E, I, H), device=dev).to(dt)
    d = torch.randn((E, H, I), device=dev).to(dt)
    off = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    xd = torch.empty((0, H), dtype=dt, device=dev)
    gg = torch.full((E, I, H), float("nan"), device=dev)
    gu = torch.full((E, I, H), float("nan"), device=dev)
    gd = torch.full((E, H, I), float("nan"), device=dev)
    moe.moe_experts_backward(xd, off, g, g, d, torch.empty(0, dtype=torch.uint8, device=dev),
                             torch.empty((0, H), dtype=dt, device=dev),
                             grad_x_disp=torch.empty((0, H), dtype=dt, device=dev),
                             grad_gate=gg, grad_up=gu, grad_down=gd)
    torch.cuda.synchronize()
    assert (gg == 0).all() and (gu == 0).all() and (gd == 0).all()


# ---------------------------------------------------------------- whole chain

CHAIN_CASES = [
    W.MoeConfig("chain_bf16", 96, T=192, H=256, I=192, E=8, top_k=2, renormalize=True,
                dtype="bf16", logits_dtype="f32"),
    W.MoeConfig("chain_f32", 97, T=96, H=128, I=64, E=4, top_k=2, renormalize=False,
                dtype="f32", logits_dtype="f32"),
]


@pytest.mark.parametrize("cfg", CHAIN_CASES, ids=lambda c: c.name)
def test_training_chain(dev, cfg):
    """Forward with a fixed selection and router weights, then the four
    backward steps in the section's order; every gradient against the oracle
    chain on the same bytes."""
    cpu = W.moe_inputs(cfg, device="cpu")
    gy = W.training_grad(cfg, device="cpu")
    on = {k: v.to(dev) for k, v in cpu.items()}
    T, k, E = cfg.T, cfg.top_k, cfg.E
    dt = on["x"].dtype
    name = cfg.dtype
    idx, _ = moe.moe_route(on["logits"], k, cfg.renormalize)
    d = moe.moe_dispatch(idx, on["x"], E)
    w = moe.moe_router_weights(on["logits"], idx, "softmax", cfg.renormalize, 1.0)
    out, cache = moe.moe_experts_forward_training(d["x_disp"], d["offsets"], on["gate"], on["up"],
                                                  on["down"], out_dtype=torch.float32)
    y = moe.moe_combine(out, w, d["row_of"], dtype=dt)
    dexp, dw = moe.moe_combine_backward(out, w, d["row_of"], gy.to(dev))
    dxd, dgate, dup, ddown = moe.moe_experts_backward(d["x_disp"], d["offsets"], on["gate"],
                                                      on["up"], on["down"], cache, dexp)
    dx = moe.moe_dispatch_backward(dxd, d["row_of"], T, k)
    dl = moe.moe_router_backward(on["logits"], idx, dw, "softmax", cfg.renormalize, 1.0)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0

    lg = np_of(cpu["logits"])
    ridx, _, _ = oracle.route(lg, "f32", k, cfg.renormalize)
    assert np.array_equal(idx.cpu().numpy().astype(np.uint32), ridx)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(ridx, E)
    rw, _ = oracle.router_weights(lg, "f32", ridx, "softmax", cfg.renormalize, 1.0, "f32")
    xd = oracle.gather(np_of(cpu["x"]), name, k, src_of, T * k)
    G, U, Dn = np_of(cpu["gate"]), np_of(cpu["up"]), np_of(cpu["down"])
    rout = oracle.experts_dispatched(xd, name, offsets, G, U, Dn)
    ry = oracle.combine(rout, "f64", rw, "f32", row_of, k)
    # the GPU's maps follow the assignment order inside each expert, as the
    # oracle's do, so they agree exactly; the gradients below use the oracle's
    assert np.array_equal(d["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(d["row_of"].cpu().numpy(), row_of)
    rdexp, rdw = oracle.combine_backward(rout, "f64", rw, "f32", row_of, np_of(gy), name, k)
    rdxd, rdg, rdu, rdd = oracle.experts_backward_dispatched(xd, name, offsets, G, U, Dn,
                                                             rdexp, "f64")
    rdx = oracle.dispatch_backward(rdxd, "f64", row_of, k)
    rdl, _ = oracle.router_backward(lg, "f32", ridx, rdw, "f64", "softmax", cfg.renormalize, 1.0,
                                    "f64")
    assert_close(to_f64(w), rw.astype(np.float64), "f32", "router weights")
    assert_close(to_f64(y), ry, name, "output")
    assert_close(to_f64(dw), rdw, name if name != "f32" else "f32", "routing-weight gradient")
    # two design roundings per product from here on (see parity.py)
    assert_close(to_f64(dx), rdx, name, "input gradient", rounds=2)
    assert_close(to_f64(dgate), rdg, name, "gate gradient", rounds=2)
    assert_close(to_f64(dup), rdu, name, "up gradient", rounds=2)
    assert_close(to_f64(ddown), rdd, name, "down gradient", rounds=2)
    assert_close(to_f64(dl), rdl, name if name != "f32" else "f32", "logits gradient")
