"""Full-size workloads, in the launch configuration the benchmark times
(``moe_forward`` with one caller workspace), against the CPU oracle.

Routing and dispatch are compared in full (they are cheap for the oracle).
Expert outputs are compared on a seeded sample of tokens that the oracle
evaluates one by one: a token's output depends only on its own row of x and
logits and on the weights of the experts it selects, so only those experts'
weights are copied to the host. The combine + Add + RMSNorm workload is
compared in full.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, per_expert_sets, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = {"fine_prefill_bf16": 24, "coarse_prefill_bf16": 4, "decode_bf16": 6}


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_forward_sampled(dev, name):
    cfg = W.CONFIGS[name]
    d = W.moe_inputs(cfg, device=dev)
    T, k, E = cfg.T, cfg.top_k, cfg.E
    ws = torch.empty(moe.moe_forward_workspace_size(T, cfg.H, cfg.I, E, k, d["x"].dtype,
                                                    d["logits"].dtype),
                     dtype=torch.uint8, device=dev)
    y = moe.moe_forward(d["x"], d["logits"], d["gate"], d["up"], d["down"], k,
                        cfg.renormalize, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0

    # routing and dispatch, in full
    logits_np, x_np = np_of(d["logits"]), np_of(d["x"])
    idx_ref, w_ref, _ = oracle.route(logits_np, cfg.logits_dtype, k, cfg.renormalize)
    idx, w = moe.moe_route(d["logits"], k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, d["x"], E)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy().view(np.uint32), idx_ref)
    assert_close(to_f64(w), oracle.to_f64(w_ref, cfg.logits_dtype), cfg.logits_dtype, "w")
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx_ref, E)
    assert np.array_equal(disp["offsets"].cpu().numpy(), offsets)
    g_src = disp["src_of"].cpu().numpy()
    assert per_expert_sets(g_src, offsets) == per_expert_sets(src_of, offsets)

    # expert outputs on sampled tokens (first, last and seeded picks)
    rng = np.random.default_rng(cfg.seed)
    n = SAMPLES[name]
    tokens = np.unique(np.concatenate([[0, T - 1], rng.choice(T, n - 2, replace=False)]))
    sel = idx_ref[tokens]                                   # [n, k]
    experts = np.unique(sel)
    remap = {int(e): i for i, e in enumerate(experts)}
    ex_t = torch.from_numpy(experts.astype(np.int64)).to(dev)
    gate = np_of(d["gate"].index_select(0, ex_t))
    up = np_of(d["up"].index_select(0, ex_t))
    down = np_of(d["down"].index_select(0, ex_t))
    rows = np.repeat(x_np[tokens], k, axis=0)
    eor = np.array([remap[int(e)] for e in sel.reshape(-1)], np.int32)
    out = oracle.swiglu_rows(rows, cfg.dtype, eor, gate, up, down)
    y_ref = oracle.combine(out, "f64", w_ref[tokens], cfg.logits_dtype,
                           np.arange(tokens.size * k, dtype=np.int32), k)
    assert_close(to_f64(y[torch.from_numpy(tokens).to(dev)]), y_ref, cfg.dtype,
                 f"{name} sampled y")
    del d, ws, y, disp
    _free()


def test_full_combine_add_rmsnorm(dev):
    cfg = W.COMBINE_NORM
    d = W.combine_norm_inputs(cfg, device=dev)
    idx, w, _ = oracle.route(np_of(d["logits"]), "f32", cfg.top_k, True)
    _, _, row_of, _, _ = oracle.dispatch(idx, cfg.E)
    w_t = torch.from_numpy(w).to(dev)
    row_t = torch.from_numpy(row_of).to(dev)
    y, x_out, rstd = moe.moe_combine_add_rmsnorm(d["out_disp"], w_t, row_t, d["residual"],
                                                 d["gamma"], cfg.eps)
    torch.cuda.synchronize()
    comb = oracle.combine(np_of(d["out_disp"]), "bf16", w, "f32", row_of, cfg.top_k)
    y_ref, x_ref, rstd_ref = oracle.add_rmsnorm(comb, np_of(d["residual"]), "bf16",
                                                np_of(d["gamma"]), "bf16", cfg.eps)
    assert_close(to_f64(x_out), oracle.to_f64(x_ref, "bf16"), "bf16", "x_out")
    assert_close(to_f64(y), oracle.to_f64(y_ref, "bf16"), "bf16", "y")
    assert_close(rstd.cpu().numpy().astype(np.float64), rstd_ref.astype(np.float64), "f32",
                 "rstd")
    del d, y, x_out
    _free()


def test_full_forward_sigmoid_grouped_sampled(dev):
    """The decode shapes with group-limited sigmoid routing (ruDNN user guide,
    section 10), through moe_forward_sigmoid_grouped: routing in full (ids
    exact outside near-ties, see test_sigmoid_grouped_gpu), y on sampled
    tokens."""
    from test_sigmoid_grouped_gpu import near_tie_rows
    cfg = W.CONFIGS["sigmoid_grouped_decode_bf16"]
    d = W.moe_inputs(cfg, device=dev)
    T, k, E = cfg.T, cfg.top_k, cfg.E
    bias = d.get("bias")
    y = moe.moe_forward_sigmoid_grouped(d["x"], d["logits"], bias, d["gate"], d["up"],
                                        d["down"], k, cfg.groups, cfg.selected_groups,
                                        cfg.group_top_two, cfg.renormalize, cfg.scale)
    idx, w = moe.moe_route_sigmoid_grouped(d["logits"], bias, k, cfg.groups,
                                           cfg.selected_groups, cfg.group_top_two,
                                           cfg.renormalize, cfg.scale)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    logits_np, x_np = np_of(d["logits"]), np_of(d["x"])
    bias_np = None if bias is None else bias.cpu().numpy()
    idx_ref, w_ref, _ = oracle.route_sigmoid_grouped(logits_np, cfg.logits_dtype, bias_np, k,
                                                     cfg.groups, cfg.selected_groups,
                                                     cfg.group_top_two, cfg.renormalize,
                                                     cfg.scale)
    skip = set(near_tie_rows(logits_np.astype(np.float32), bias_np, k, cfg.groups,
                             cfg.selected_groups, cfg.group_top_two))
    assert len(skip) <= 2
    keep = np.array([t for t in range(T) if t not in skip])
    assert np.array_equal(idx.cpu().numpy().view(np.uint32)[keep], idx_ref[keep])
    assert_close(to_f64(w)[keep], oracle.to_f64(w_ref, cfg.logits_dtype)[keep],
                 cfg.logits_dtype, "w")

    rng = np.random.default_rng(cfg.seed)
    tokens = np.array(sorted(set(rng.choice(keep, 8, replace=False).tolist()) | {int(keep[0])}))
    sel = idx_ref[tokens]
    experts = np.unique(sel)
    remap = {int(e): i for i, e in enumerate(experts)}
    ex_t = torch.from_numpy(experts.astype(np.int64)).to(dev)
    gate = np_of(d["gate"].index_select(0, ex_t))
    up = np_of(d["up"].index_select(0, ex_t))
    down = np_of(d["down"].index_select(0, ex_t))
    rows = np.repeat(x_np[tokens], k, axis=0)
    eor = np.array([remap[int(e)] for e in sel.reshape(-1)], np.int32)
    out = oracle.swiglu_rows(rows, cfg.dtype, eor, gate, up, down)
    y_ref = oracle.combine(out, "f64", w_ref[tokens], cfg.logits_dtype,
                           np.arange(tokens.size * k, dtype=np.int32), k)
    assert_close(to_f64(y[torch.from_numpy(tokens).to(dev)]), y_ref, cfg.dtype,
                 "sigmoid-routed sampled y")
    del d, y
    _free()
