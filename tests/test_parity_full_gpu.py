"""Full-size workloads, in the launch configuration the benchmark times
(``moe_forward`` with one caller workspace), against the CPU oracle.

For the fine prefill, coarse prefill and decode workloads:

* the routing plan and dispatch map that the one-call forward itself left in
  its workspace (ids, weights, counts, offsets, row_of, src_of; located with
  moe_forward_workspace_layout) are compared in full with the oracle's: ids,
  counts, offsets and maps bit for bit, weights within the bar;
* y is compared on tokens the oracle evaluates one by one, chosen from the
  oracle's dispatch map so that every expert's first, middle and last
  M-tile units of the tile schedule are hit (the first and last rows of each
  CTA's half of a unit), plus seeded picks; the decode workload is compared
  on all of its tokens. A token's output depends only on its own row of x
  and logits and on the weights of the experts it selects, so only those
  experts' weights are copied to the host;
* guard bands before and after y and the workspace stay untouched.

The combine + Add + RMSNorm workload is compared in full.
"""

from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import assert_close, np_of, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GUARD = 4096
GUARD_BYTE = 0xA5
PAIR_ROWS = 256          # rows of one CTA-pair unit of the expert GEMMs
CTA_ROWS = 128           # rows of one CTA's half of a unit

# tokens compared per workload: "all", or at least this many
SAMPLES = {"fine_prefill_bf16": 128, "coarse_prefill_bf16": 64, "decode_bf16": "all"}


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


def guarded(nbytes: int, dev):
    whole = torch.full((nbytes + 2 * GUARD,), GUARD_BYTE, dtype=torch.uint8, device=dev)
    return whole, whole[GUARD:GUARD + nbytes]


def assert_guards_intact(whole: torch.Tensor, what: str):
    assert bool(torch.all(whole[:GUARD] == GUARD_BYTE)), f"{what}: guard before written"
    assert bool(torch.all(whole[-GUARD:] == GUARD_BYTE)), f"{what}: guard after written"


def plan_view(ws, lay, T, k, E, ldt):
    A = T * k

    def view(off, n, dt):
        return ws[off:off + n * torch.tensor([], dtype=dt).element_size()].view(dt)
    return {"idx": view(lay["expert_indices"], A, torch.int32).reshape(T, k),
            "w": view(lay["weights"], A, ldt).reshape(T, k),
            "counts": view(lay["counts"], E, torch.int32),
            "offsets": view(lay["offsets"], E + 1, torch.int32),
            "row_of": view(lay["row_of"], A, torch.int32),
            "src_of": view(lay["src_of"], A, torch.int32)}


def schedule_rows(seg: int) -> list[int]:
    """Rows inside an expert's segment at the edges of its first, middle and
    last CTA-pair units: the first and last row of each CTA's 128-row half
    (an expert's last unit with at most 128 rows runs as one M = 128 tile)."""
    if seg <= 0:
        return []
    units = (seg + PAIR_ROWS - 1) // PAIR_ROWS
    picks = set()
    for j in {0, units // 2, units - 1}:
        base = j * PAIR_ROWS
        for r in (base, base + CTA_ROWS - 1, base + CTA_ROWS, base + PAIR_ROWS - 1):
            if r < seg:
                picks.add(r)
    picks.add(seg - 1)
    return sorted(picks)


def sample_tokens(name, T, k, offsets, src_of, seed):
    want = SAMPLES[name]
    if want == "all":
        return np.arange(T)
    toks = set()
    for e in range(len(offsets) - 1):
        seg = int(offsets[e + 1] - offsets[e])
        for r in schedule_rows(seg):
            toks.add(int(src_of[offsets[e] + r]) // k)
    toks |= {0, T - 1}
    rng = np.random.default_rng(seed)
    while len(toks) < want:
        toks.add(int(rng.integers(T)))
    return np.array(sorted(toks))


def swiglu_rows_threaded(rows, dt, eor, gate, up, down):
    """oracle.swiglu_rows over row chunks on every host core (the C oracle
    runs without the GIL); each row's result is the oracle's own."""
    n = rows.shape[0]
    threads = max(1, min(os.cpu_count() or 1, n))
    bounds = np.linspace(0, n, threads + 1).astype(int)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda i: oracle.swiglu_rows(rows[bounds[i]:bounds[i + 1]], dt,
                                                         eor[bounds[i]:bounds[i + 1]], gate, up,
                                                         down),
                            range(threads)))
    return np.concatenate(parts, axis=0)


@pytest.mark.parametrize("name", list(SAMPLES))
def test_full_forward(dev, name):
    cfg = W.CONFIGS[name]
    d = W.moe_inputs(cfg, device=dev)
    T, H, k, E = cfg.T, cfg.H, cfg.top_k, cfg.E
    lay = moe.moe_forward_workspace_layout(T, H, cfg.I, E, k, d["x"].dtype, d["logits"].dtype)
    ws_whole, ws = guarded(lay["total"], dev)
    y_whole, y_bytes = guarded(T * H * d["x"].element_size(), dev)
    y = y_bytes.view(d["x"].dtype).view(T, H)
    moe.moe_forward(d["x"], d["logits"], d["gate"], d["up"], d["down"], k, cfg.renormalize,
                    y=y, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert_guards_intact(ws_whole, f"{name} workspace")
    assert_guards_intact(y_whole, f"{name} y")

    # the forward's own routing plan and dispatch map, in full
    logits_np, x_np = np_of(d["logits"]), np_of(d["x"])
    idx_ref, w_ref, _ = oracle.route(logits_np, cfg.logits_dtype, k, cfg.renormalize)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx_ref, E)
    plan = plan_view(ws, lay, T, k, E, d["logits"].dtype)
    assert np.array_equal(plan["idx"].cpu().numpy().view(np.uint32), idx_ref), "ids"
    assert_close(to_f64(plan["w"]), oracle.to_f64(w_ref, cfg.logits_dtype), cfg.logits_dtype,
                 f"{name} weights")
    assert np.array_equal(plan["counts"].cpu().numpy(), counts), "counts"
    assert np.array_equal(plan["offsets"].cpu().numpy(), offsets), "offsets"
    assert np.array_equal(plan["row_of"].cpu().numpy(), row_of), "row_of"
    assert np.array_equal(plan["src_of"].cpu().numpy(), src_of), "src_of"

    # expert outputs on tokens covering the tile schedule of every expert
    tokens = sample_tokens(name, T, k, offsets, src_of, cfg.seed)
    assert tokens.size >= (T if SAMPLES[name] == "all" else SAMPLES[name])
    sel = idx_ref[tokens]                                   # [n, k]
    experts = np.unique(sel)
    remap = {int(e): i for i, e in enumerate(experts)}
    ex_t = torch.from_numpy(experts.astype(np.int64)).to(dev)
    gate = np_of(d["gate"].index_select(0, ex_t))
    up = np_of(d["up"].index_select(0, ex_t))
    down = np_of(d["down"].index_select(0, ex_t))
    rows = np.repeat(x_np[tokens], k, axis=0)
    eor = np.array([remap[int(e)] for e in sel.reshape(-1)], np.int32)
    out = swiglu_rows_threaded(rows, cfg.dtype, eor, gate, up, down)
    y_ref = oracle.combine(out, "f64", w_ref[tokens], cfg.logits_dtype,
                           np.arange(tokens.size * k, dtype=np.int32), k)
    assert_close(to_f64(y[torch.from_numpy(tokens).to(dev)]), y_ref, cfg.dtype,
                 f"{name} y on {tokens.size} tokens")
    del d, ws, ws_whole, y, y_whole
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


def test_full_forward_sigmoid_grouped(dev):
    """The decode shapes with group-limited sigmoid routing (ruDNN user guide,
    section 10), through moe_forward_sigmoid_grouped: the routing the forward
    kept in its workspace bit for bit on every row, y on sampled tokens."""
    cfg = W.CONFIGS["sigmoid_grouped_decode_bf16"]
    d = W.moe_inputs(cfg, device=dev)
    T, k, E = cfg.T, cfg.top_k, cfg.E
    bias = d.get("bias")
    lay = moe.moe_forward_workspace_layout(T, cfg.H, cfg.I, E, k, d["x"].dtype,
                                           d["logits"].dtype)
    ws = torch.empty(lay["total"], dtype=torch.uint8, device=dev)
    y = moe.moe_forward_sigmoid_grouped(d["x"], d["logits"], bias, d["gate"], d["up"],
                                        d["down"], k, cfg.groups, cfg.selected_groups,
                                        cfg.group_top_two, cfg.renormalize, cfg.scale,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    logits_np, x_np = np_of(d["logits"]), np_of(d["x"])
    bias_np = None if bias is None else bias.cpu().numpy()
    idx_ref, w_ref, _ = oracle.route_sigmoid_grouped(logits_np, cfg.logits_dtype, bias_np, k,
                                                     cfg.groups, cfg.selected_groups,
                                                     cfg.group_top_two, cfg.renormalize,
                                                     cfg.scale)
    plan = plan_view(ws, lay, T, k, E, d["logits"].dtype)
    assert np.array_equal(plan["idx"].cpu().numpy().view(np.uint32), idx_ref)
    assert_close(to_f64(plan["w"]), oracle.to_f64(w_ref, cfg.logits_dtype), cfg.logits_dtype,
                 "w")
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx_ref, E)
    assert np.array_equal(plan["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(plan["row_of"].cpu().numpy(), row_of)

    rng = np.random.default_rng(cfg.seed)
    tokens = np.array(sorted(set(rng.choice(T, 16, replace=False).tolist()) | {0, T - 1}))
    sel = idx_ref[tokens]
    experts = np.unique(sel)
    remap = {int(e): i for i, e in enumerate(experts)}
    ex_t = torch.from_numpy(experts.astype(np.int64)).to(dev)
    gate = np_of(d["gate"].index_select(0, ex_t))
    up = np_of(d["up"].index_select(0, ex_t))
    down = np_of(d["down"].index_select(0, ex_t))
    rows = np.repeat(x_np[tokens], k, axis=0)
    eor = np.array([remap[int(e)] for e in sel.reshape(-1)], np.int32)
    out = swiglu_rows_threaded(rows, cfg.dtype, eor, gate, up, down)
    y_ref = oracle.combine(out, "f64", w_ref[tokens], cfg.logits_dtype,
                           np.arange(tokens.size * k, dtype=np.int32), k)
    assert_close(to_f64(y[torch.from_numpy(tokens).to(dev)]), y_ref, cfg.dtype,
                 "sigmoid-routed sampled y")
    del d, y, ws
    _free()
