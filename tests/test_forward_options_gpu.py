"""moe_forward_ex: the one-call forward (ruDNN user guide, section 6) with its
options, against the CPU oracle and against itself.

* MOE_FORWARD_DETERMINISTIC: the combine runs as the slot-order kernel over
  FP32 expert outputs, so two calls on the same inputs give the same bits
  (the default BF16/F16 forward adds its rows in arrival order);
* group-limited sigmoid routing (ruDNN user guide, section 10) selected
  through the options computes what moe_forward_sigmoid_grouped computes;
* events around the expert GEMMs change nothing in the result;
* the saved routing plan and dispatch map the forward leaves in its
  workspace (moe_forward_workspace_layout) equal the oracle's, bit for bit;
* guard bands around y and the workspace stay untouched.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, to_f64

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of guard band on each side (keeps 256-byte alignment)
GUARD_BYTE = 0xA5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def guarded(nbytes: int, dev):
    """A byte buffer with GUARD bytes of GUARD_BYTE on each side of its
    nbytes interior; returns (whole, interior)."""
    whole = torch.full((nbytes + 2 * GUARD,), GUARD_BYTE, dtype=torch.uint8, device=dev)
    return whole, whole[GUARD:GUARD + nbytes]


def assert_guards_intact(whole: torch.Tensor, what: str):
    head, tail = whole[:GUARD], whole[-GUARD:]
    assert bool(torch.all(head == GUARD_BYTE)), f"{what}: guard band before the buffer written"
    assert bool(torch.all(tail == GUARD_BYTE)), f"{what}: guard band after the buffer written"


def workspace_plan(ws: torch.Tensor, lay: dict, T: int, k: int, E: int, ldt: torch.dtype):
    """The routing plan and dispatch map the forward left in its workspace."""
    A = T * k

    def view(off, n, dt):
        return ws[off:off + n * torch.tensor([], dtype=dt).element_size()].view(dt)
    return {"idx": view(lay["expert_indices"], A, torch.int32).reshape(T, k),
            "w": view(lay["weights"], A, ldt).reshape(T, k),
            "counts": view(lay["counts"], E, torch.int32),
            "offsets": view(lay["offsets"], E + 1, torch.int32),
            "row_of": view(lay["row_of"], A, torch.int32),
            "src_of": view(lay["src_of"], A, torch.int32)}


def assert_plan_matches_oracle(plan, cfg, logits_np, what):
    """Ids, counts, offsets and both maps bit-exact (the GPU orders an
    expert's rows by assignment, as the oracle's stable dispatch does);
    weights within the bar of the logits dtype."""
    T, k, E = cfg.T, cfg.top_k, cfg.E
    idx_ref, w_ref, _ = oracle.route(logits_np, cfg.logits_dtype, k, cfg.renormalize)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx_ref, E)
    assert np.array_equal(plan["idx"].cpu().numpy().view(np.uint32), idx_ref), f"{what}: ids"
    assert_close(to_f64(plan["w"]), oracle.to_f64(w_ref, cfg.logits_dtype), cfg.logits_dtype,
                 f"{what}: weights")
    assert np.array_equal(plan["counts"].cpu().numpy(), counts), f"{what}: counts"
    assert np.array_equal(plan["offsets"].cpu().numpy(), offsets), f"{what}: offsets"
    assert np.array_equal(plan["row_of"].cpu().numpy(), row_of), f"{what}: row_of"
    assert np.array_equal(plan["src_of"].cpu().numpy(), src_of), f"{what}: src_of"
    return idx_ref, w_ref, offsets, src_of


CASES = [
    # folded combine by default (T*H*4 <= 64 MiB), CTA pairs (>= 256 rows per expert)
    W.MoeConfig("opt_pair_bf16", 92, T=1024, H=256, I=192, E=4, top_k=2, renormalize=True,
                dtype="bf16", logits_dtype="f32", logit_bias="normal", bias_param=0.5),
    # single CTAs, many experts, BF16 logits, no renormalisation
    W.MoeConfig("opt_many_bf16", 93, T=300, H=128, I=136, E=64, top_k=6, renormalize=False,
                dtype="bf16", logits_dtype="bf16"),
    W.MoeConfig("opt_f16", 94, T=200, H=192, I=96, E=8, top_k=3, renormalize=True,
                dtype="f16", logits_dtype="f16"),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_deterministic_forward_is_bit_reproducible(dev, cfg):
    g = {n: v.to(dev) for n, v in W.moe_inputs(cfg, device="cpu").items()}
    o = {n: np_of(v.cpu()) for n, v in g.items()}
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"], o["up"],
                         o["down"], cfg.top_k, cfg.renormalize)
    ys = []
    for _ in range(3):
        ys.append(moe.moe_forward_ex(g["x"], g["logits"], g["gate"], g["up"], g["down"],
                                     cfg.top_k, cfg.renormalize, deterministic=True))
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    assert torch.equal(ys[0].view(torch.int16), ys[2].view(torch.int16))
    assert_close(to_f64(ys[0]), ref["y"], cfg.dtype, f"{cfg.name} deterministic y")
    # the staged calls run the same slot-order combine over FP32 expert
    # outputs: the result is within the bar as well
    idx, w = moe.moe_route(g["logits"], cfg.top_k, cfg.renormalize)
    d = moe.moe_dispatch(idx, g["x"], cfg.E)
    out = moe.moe_experts_forward(d["x_disp"], d["offsets"], g["gate"], g["up"], g["down"],
                                  out_dtype=torch.float32)
    y2 = moe.moe_combine(out, w, d["row_of"], dtype=g["x"].dtype)
    torch.cuda.synchronize()
    assert_close(to_f64(y2), ref["y"], cfg.dtype, f"{cfg.name} staged y")


@pytest.mark.parametrize("deterministic", [False, True], ids=["folded", "deterministic"])
@pytest.mark.parametrize("cfg", CASES[:2], ids=lambda c: c.name)
def test_forward_plan_in_workspace_and_guards(dev, cfg, deterministic):
    """The workspace regions moe_forward_workspace_layout names hold the
    routing plan and dispatch map, equal to the oracle's; nothing is written
    outside y or outside the workspace's total bytes; events around the
    expert GEMMs measure a positive time."""
    g = {n: v.to(dev) for n, v in W.moe_inputs(cfg, device="cpu").items()}
    T, H, k, E = cfg.T, cfg.H, cfg.top_k, cfg.E
    lay = moe.moe_forward_workspace_layout(T, H, cfg.I, E, k, g["x"].dtype, g["logits"].dtype,
                                           deterministic)
    ws_whole, ws = guarded(lay["total"], dev)
    y_whole, y_bytes = guarded(T * H * g["x"].element_size(), dev)
    y = y_bytes.view(g["x"].dtype).view(T, H)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    moe.moe_forward_ex(g["x"], g["logits"], g["gate"], g["up"], g["down"], k, cfg.renormalize,
                       deterministic=deterministic, experts_begin_event=ev0,
                       experts_end_event=ev1, y=y, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert ev0.elapsed_time(ev1) > 0.0
    assert_guards_intact(ws_whole, "workspace")
    assert_guards_intact(y_whole, "y")
    plan = workspace_plan(ws, lay, T, k, E, g["logits"].dtype)
    logits_np = np_of(g["logits"].cpu())
    assert_plan_matches_oracle(plan, cfg, logits_np, cfg.name)
    o = {n: np_of(v.cpu()) for n, v in g.items()}
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"], o["up"],
                         o["down"], k, cfg.renormalize)
    assert_close(to_f64(y), ref["y"], cfg.dtype, f"{cfg.name} y")


def test_forward_ex_sigmoid_grouped(dev):
    """Group-limited sigmoid routing through the options: the result of
    moe_forward_sigmoid_grouped, deterministic here, against the oracle."""
    cfg = W.MoeConfig("opt_sg_bf16", 95, T=400, H=256, I=128, E=64, top_k=6, renormalize=True,
                      dtype="bf16", logits_dtype="f32")
    g = {n: v.to(dev) for n, v in W.moe_inputs(cfg, device="cpu").items()}
    gen = torch.Generator().manual_seed(7)
    bias = (torch.randn((cfg.E,), generator=gen) * 0.1).to(dev)
    sg = {"bias": bias, "groups": 8, "selected_groups": 3, "group_top_two": True, "scale": 2.5}
    ys = [moe.moe_forward_ex(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                             cfg.renormalize, deterministic=True, sigmoid_grouped=sg)
          for _ in range(2)]
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert torch.equal(ys[0].view(torch.int16), ys[1].view(torch.int16))
    o = {n: np_of(v.cpu()) for n, v in g.items()}
    ref = oracle.forward_sigmoid_grouped(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype,
                                         bias.cpu().numpy(), o["gate"], o["up"], o["down"],
                                         cfg.top_k, 8, 3, True, True, 2.5)
    assert_close(to_f64(ys[0]), ref["y"], cfg.dtype, "sigmoid-routed deterministic y")
    # and the routing the forward kept equals the oracle's, bit for bit
    lay = moe.moe_forward_workspace_layout(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k,
                                           g["x"].dtype, g["logits"].dtype, True)
    ws = torch.empty(lay["total"], dtype=torch.uint8, device=dev)
    moe.moe_forward_ex(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                       cfg.renormalize, deterministic=True, sigmoid_grouped=sg, workspace=ws)
    torch.cuda.synchronize()
    plan = workspace_plan(ws, lay, cfg.T, cfg.top_k, cfg.E, g["logits"].dtype)
    assert np.array_equal(plan["idx"].cpu().numpy().view(np.uint32), ref["idx"])
