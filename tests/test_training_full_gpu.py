"""The training step at full size (the fine and the coarse prefill's shapes,
the launch configurations ``bench.py --workload train_fine_prefill_bf16`` and
``train_coarse_prefill_bf16`` time) against the CPU oracle (ruDNN user guide,
section 12).

The GPU runs the whole chain: route, dispatch, router weights, the training
forward, combine, then the combine, expert, dispatch and router backward.
The oracle checks what it can compute piecewise:

* the input and logits gradients of a seeded sample of tokens: a token's
  gradients depend only on its own rows (its x, logits and output gradient)
  and on the weights of the experts it selects;
* the full FP32 gate / up / down gradients of one expert (the one with the
  fewest rows, to keep the oracle's double loops short), which sum over every
  row the expert received; on the coarse shapes (58.7 M weights per matrix)
  the gradients of two experts at sampled intermediate columns instead.

Bars: the chained backward's (two design roundings per product, ``parity``)
for the input and weight gradients; the BF16 bar for the logits gradient.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE_TOKENS = 8


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def _one_expert(w, e):
    """Expert e's weights as a one-expert stack, in oracle storage."""
    return np.ascontiguousarray(np_of(w[e:e + 1]))


def test_training_step_full_size(dev):
    cfg = W.CONFIGS["fine_prefill_bf16"]
    d = W.moe_inputs(cfg, device=dev)
    gy = W.training_grad(cfg, device=dev)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    name, lname = cfg.dtype, cfg.logits_dtype

    idx, _ = moe.moe_route(d["logits"], k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, d["x"], E)
    w = moe.moe_router_weights(d["logits"], idx, "softmax", cfg.renormalize, 1.0)
    out, cache = moe.moe_experts_forward_training(disp["x_disp"], disp["offsets"], d["gate"],
                                                  d["up"], d["down"], out_dtype=torch.float32)
    dexp, dw = moe.moe_combine_backward(out, w, disp["row_of"], gy)
    dxd, dgate, dup, ddown = moe.moe_experts_backward(disp["x_disp"], disp["offsets"],
                                                      d["gate"], d["up"], d["down"], cache, dexp)
    dx = moe.moe_dispatch_backward(dxd, disp["row_of"], T, k)
    dl = moe.moe_router_backward(d["logits"], idx, dw, "softmax", cfg.renormalize, 1.0)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0

    logits_np, x_np, gy_np = np_of(d["logits"]), np_of(d["x"]), np_of(gy)
    ridx, _, _ = oracle.route(logits_np, lname, k, cfg.renormalize)
    assert np.array_equal(idx.cpu().numpy().astype(np.uint32), ridx)

    # sampled tokens: every slot's expert evaluated on that token's row alone
    rng = np.random.default_rng(cfg.seed + 77)
    tokens = rng.choice(T, size=SAMPLE_TOKENS, replace=False)
    rdx = np.zeros((SAMPLE_TOKENS, H))
    rdw = np.zeros((SAMPLE_TOKENS, k))
    lg_s = np.ascontiguousarray(logits_np[tokens])
    rw, _ = oracle.router_weights(lg_s, lname, ridx[tokens], "softmax", cfg.renormalize, 1.0, "f32")
    for i, t in enumerate(tokens):
        xrow = np.ascontiguousarray(x_np[t:t + 1])
        for j in range(k):
            e = int(ridx[t, j])
            G, U, D = (_one_expert(d[n], e) for n in ("gate", "up", "down"))
            o = oracle.swiglu_rows(xrow, name, np.zeros(1, np.int32), G, U, D)
            rdw[i, j] = float(np.dot(oracle.to_f64(gy_np[t], name), o[0]))
            dexp_row = float(rw[i, j]) * oracle.to_f64(gy_np[t:t + 1], name)
            rdx[i] += oracle.swiglu_backward_rows(xrow, name, np.zeros(1, np.int32), G, U, D,
                                                  dexp_row, "f64")[0][0]
    rdl, _ = oracle.router_backward(lg_s, lname, ridx[tokens], rdw, "f64", "softmax",
                                    cfg.renormalize, 1.0, "f64")
    assert_close(to_f64(dw)[tokens], rdw, name, "routing-weight gradient (sampled)")
    assert_close(to_f64(dx)[tokens], rdx, name, "input gradient (sampled)", rounds=2)
    assert_close(to_f64(dl)[tokens], rdl, lname if lname != "f32" else "f32",
                 "logits gradient (sampled)")

    # one expert's full weight gradients (all of its rows, from the oracle's
    # own dispatch, which the GPU's matches exactly)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(ridx, E)
    assert np.array_equal(disp["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(disp["src_of"].cpu().numpy(), src_of)
    e = int(np.argmin(np.where(counts > 0, counts, np.iinfo(np.int32).max)))
    src = src_of[offsets[e]:offsets[e + 1]]
    toks, slots = src // k, src % k
    rw_e, _ = oracle.router_weights(np.ascontiguousarray(logits_np[toks]), lname, ridx[toks],
                                    "softmax", cfg.renormalize, 1.0, "f64")
    dexp_e = rw_e[np.arange(toks.size), slots][:, None] * oracle.to_f64(gy_np[toks], name)
    G, U, D = (_one_expert(d[n], e) for n in ("gate", "up", "down"))
    _, rg, ru, rd = oracle.swiglu_backward_rows(np.ascontiguousarray(x_np[toks]), name,
                                                np.zeros(toks.size, np.int32), G, U, D,
                                                np.ascontiguousarray(dexp_e), "f64")
    assert_close(to_f64(dgate[e]), rg[0], name, f"gate gradient of expert {e}", rounds=2)
    assert_close(to_f64(dup[e]), ru[0], name, f"up gradient of expert {e}", rounds=2)
    assert_close(to_f64(ddown[e]), rd[0], name, f"down gradient of expert {e}", rounds=2)


# ------------------------------------------------ coarse prefill shapes, full size

COARSE_COLS = (0, 127, 128, 255, 256, 7167, 14335)   # intermediate columns sampled


def _columns_of_expert(w_gate, w_up, w_down, e, cols):
    """Expert e restricted to the intermediate columns `cols`: rows of its gate
    and up weights and columns of its down weight, as a one-expert stack. In a
    SwiGLU FFN each intermediate column i touches only row i of Wg / Wu and
    column i of Wd, so the backward of this restricted expert gives exactly the
    full expert's weight gradients at those columns."""
    c = torch.as_tensor(cols, device=w_gate.device)
    G = np.ascontiguousarray(np_of(w_gate[e:e + 1, c, :]))
    U = np.ascontiguousarray(np_of(w_up[e:e + 1, c, :]))
    D = np.ascontiguousarray(np_of(w_down[e:e + 1][:, :, c]))
    return G, U, D


def test_training_step_coarse_full_size(dev):
    """The training step on the coarse prefill's shapes (the launch
    configuration ``bench.py --workload train_coarse_prefill_bf16`` times:
    4096 rows per expert, so the expert backward runs on CTA pairs): routing
    bit-exact, sampled tokens' input, routing-weight and logits gradients, and
    the weight gradients of the smallest and the largest expert at sampled
    intermediate columns (both halves of a pair's M = 256 tile and its
    edges, the middle and the last column), each over all of that expert's
    rows."""
    cfg = W.CONFIGS["coarse_prefill_bf16"]
    d = W.moe_inputs(cfg, device=dev)
    gy = W.training_grad(cfg, device=dev)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    name, lname = cfg.dtype, cfg.logits_dtype
    assert T * k >= 2048 * E                              # the pair mode's condition

    idx, _ = moe.moe_route(d["logits"], k, cfg.renormalize)
    disp = moe.moe_dispatch(idx, d["x"], E)
    w = moe.moe_router_weights(d["logits"], idx, "softmax", cfg.renormalize, 1.0)
    out, cache = moe.moe_experts_forward_training(disp["x_disp"], disp["offsets"], d["gate"],
                                                  d["up"], d["down"], out_dtype=torch.float32)
    dexp, dw = moe.moe_combine_backward(out, w, disp["row_of"], gy)
    dxd, dgate, dup, ddown = moe.moe_experts_backward(disp["x_disp"], disp["offsets"],
                                                      d["gate"], d["up"], d["down"], cache, dexp)
    dx = moe.moe_dispatch_backward(dxd, disp["row_of"], T, k)
    dl = moe.moe_router_backward(d["logits"], idx, dw, "softmax", cfg.renormalize, 1.0)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0

    logits_np, x_np, gy_np = np_of(d["logits"]), np_of(d["x"]), np_of(gy)
    ridx, _, _ = oracle.route(logits_np, lname, k, cfg.renormalize)
    assert np.array_equal(idx.cpu().numpy().astype(np.uint32), ridx)

    # sampled tokens, as on the fine prefill's shapes
    rng = np.random.default_rng(cfg.seed + 78)
    n_tok = 4
    tokens = rng.choice(T, size=n_tok, replace=False)
    rdx = np.zeros((n_tok, H))
    rdw = np.zeros((n_tok, k))
    lg_s = np.ascontiguousarray(logits_np[tokens])
    rw, _ = oracle.router_weights(lg_s, lname, ridx[tokens], "softmax", cfg.renormalize, 1.0, "f32")
    for i, t in enumerate(tokens):
        xrow = np.ascontiguousarray(x_np[t:t + 1])
        for j in range(k):
            e = int(ridx[t, j])
            G, U, D = (_one_expert(d[n], e) for n in ("gate", "up", "down"))
            o = oracle.swiglu_rows(xrow, name, np.zeros(1, np.int32), G, U, D)
            rdw[i, j] = float(np.dot(oracle.to_f64(gy_np[t], name), o[0]))
            dexp_row = float(rw[i, j]) * oracle.to_f64(gy_np[t:t + 1], name)
            rdx[i] += oracle.swiglu_backward_rows(xrow, name, np.zeros(1, np.int32), G, U, D,
                                                  dexp_row, "f64")[0][0]
            del G, U, D
    rdl, _ = oracle.router_backward(lg_s, lname, ridx[tokens], rdw, "f64", "softmax",
                                    cfg.renormalize, 1.0, "f64")
    assert_close(to_f64(dw)[tokens], rdw, name, "routing-weight gradient (sampled)")
    assert_close(to_f64(dx)[tokens], rdx, name, "input gradient (sampled)", rounds=2)
    # the logits are FP32 here, but their gradient is linear in the
    # routing-weight gradients, which come from the BF16 expert outputs: it
    # takes their bar
    assert_close(to_f64(dl)[tokens], rdl, name, "logits gradient (sampled)")

    # weight gradients at sampled columns of the smallest and the largest
    # expert, over all of their rows (from the oracle's own dispatch, which
    # the GPU's matches exactly)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(ridx, E)
    assert np.array_equal(disp["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(disp["src_of"].cpu().numpy(), src_of)
    cols = list(COARSE_COLS)
    for e in (int(np.argmin(counts)), int(np.argmax(counts))):
        src = src_of[offsets[e]:offsets[e + 1]]
        toks, slots = src // k, src % k
        rw_e, _ = oracle.router_weights(np.ascontiguousarray(logits_np[toks]), lname, ridx[toks],
                                        "softmax", cfg.renormalize, 1.0, "f64")
        dexp_e = rw_e[np.arange(toks.size), slots][:, None] * oracle.to_f64(gy_np[toks], name)
        G, U, D = _columns_of_expert(d["gate"], d["up"], d["down"], e, cols)
        _, rg, ru, rd = oracle.swiglu_backward_rows(np.ascontiguousarray(x_np[toks]), name,
                                                    np.zeros(toks.size, np.int32), G, U, D,
                                                    np.ascontiguousarray(dexp_e), "f64")
        c = torch.as_tensor(cols, device=dev)
        assert_close(to_f64(dgate[e][c, :]), rg[0], name,
                     f"gate gradient of expert {e} ({counts[e]} rows), sampled rows", rounds=2)
        assert_close(to_f64(dup[e][c, :]), ru[0], name,
                     f"up gradient of expert {e}, sampled rows", rounds=2)
        assert_close(to_f64(ddown[e][:, c]), rd[0], name,
                     f"down gradient of expert {e}, sampled columns", rounds=2)
