"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Every input is seeded and synthetic (``workloads``); every expected value
comes from ``oracle/`` on the same bytes. Sizes span several 128-row tiles,
ragged K/N/M edges, empty experts and the degenerate cases (E=1, top_k=E,
invalid rows, T=0). Full-size workloads are checked in
``test_parity_full_gpu.py``.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_topk_gb300 as moe
from mixture_experts_ffn_topk_gb300 import workloads as W
from parity import TORCH_TO_NAME, assert_close, np_of, per_expert_sets, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_topk_gb300 import build
    build.build()
    moe.load_library()
    return torch.device("cuda:0")


def cfg_small(name, **kw):
    return W.MoeConfig(name, 90, **kw)


# (name, T, H, I, E, k, renorm, dtype, logits dtype, bias, bias param)
SMALL = [
    cfg_small("multi_tile_bf16", T=300, H=320, I=200, E=6, top_k=2, renormalize=True,
              dtype="bf16", logits_dtype="f32", logit_bias="normal", bias_param=1.0),
    cfg_small("many_experts_bf16", T=256, H=256, I=136, E=64, top_k=6,
              renormalize=False, dtype="bf16", logits_dtype="bf16"),
    cfg_small("single_expert_bf16", T=150, H=192, I=264, E=1, top_k=1,
              renormalize=True, dtype="bf16", logits_dtype="bf16"),
    cfg_small("topk_equals_e_f16", T=70, H=128, I=64, E=4, top_k=4, renormalize=True,
              dtype="f16", logits_dtype="f16"),
    cfg_small("hot_expert_bf16", T=400, H=128, I=128, E=8, top_k=2, renormalize=True,
              dtype="bf16", logits_dtype="f32", logit_bias="zipf", bias_param=3.0),
    cfg_small("multi_tile_f32", T=200, H=192, I=136, E=5, top_k=2, renormalize=False,
              dtype="f32", logits_dtype="f32", logit_bias="normal", bias_param=0.5),
    W.CONFIGS["tiny_fp32"],
    # at least 2 x 128 rows per expert on average: the expert GEMMs run on CTA
    # pairs (one 256-row M-tile over two SMs); odd M-tile counts per expert
    # (3/5/1 and 3/3/3/3 here) leave the second CTA of a pair past the rows,
    # H = 200 leaves a K tail, I = 200 a partial N tile
    cfg_small("pair_skewed_bf16", T=900, H=200, I=200, E=3, top_k=1, renormalize=False,
              dtype="bf16", logits_dtype="bf16", logit_bias="zipf", bias_param=1.0),
    cfg_small("pair_f16", T=640, H=384, I=320, E=4, top_k=2, renormalize=True,
              dtype="f16", logits_dtype="f32"),
    # at least 2048 rows per expert on average: pairs with two k-blocks per
    # pipeline stage (H = 256: four k-blocks, I = 192: three, the last stage
    # of each GEMM2 unit half past K); in the one-call forward the folded
    # combine's per-expert handoff runs in this mode too
    cfg_small("pair_two_kb_bf16", T=4400, H=256, I=192, E=2, top_k=1, renormalize=True,
              dtype="bf16", logits_dtype="f32", logit_bias="normal", bias_param=0.5),
]
PAIR = [c for c in SMALL if c.name.startswith("pair_")]


def oracle_inputs(d):
    return {k: np_of(v) for k, v in d.items()}


def inputs_on(cfg, dev):
    cpu = W.moe_inputs(cfg, device="cpu")
    return cpu, {k: v.to(dev) for k, v in cpu.items()}


# ---------------------------------------------------------------- routing

ROUTE_CASES = [
    # (T, E, k, renorm, logits dtype, generator)
    (1000, 64, 6, False, "bf16", "normal"),
    (1000, 8, 2, True, "f32", "normal"),
    (333, 256, 8, True, "f32", "normal"),
    (257, 33, 5, True, "f16", "normal"),
    (64, 1, 1, False, "f32", "normal"),
    (64, 1, 1, True, "bf16", "normal"),
    (50, 7, 7, True, "f32", "normal"),
    (40, 1024, 16, True, "f32", "normal"),
    (12, 1024, 1024, False, "f32", "normal"),
    (500, 16, 4, True, "f32", "ties"),
    (500, 40, 3, False, "bf16", "ties"),
    (300, 24, 4, True, "f32", "specials"),
    # T >= 64 tokens per SM: one thread routes one token (E <= 64, k <= 8);
    # 16-byte row loads where E * dtype size % 16 == 0
    (100000, 64, 6, False, "bf16", "normal"),
    (90000, 8, 2, True, "f32", "ties"),
    (80000, 33, 5, True, "f16", "specials"),
    (80000, 24, 8, True, "bf16", "ties"),
    (100000, 64, 8, True, "f32", "specials"),
    (12000, 40, 3, False, "bf16", "ties"),
    # 16-bit logits with E % 8 == 0 at that T: the packed-pair kernel (rows
    # padded to 8 / 16 / 32 / 64 logits with -inf where E is smaller)
    (60000, 64, 8, True, "bf16", "specials"),
    (50000, 16, 4, False, "f16", "specials"),
    (40000, 48, 6, True, "f16", "ties"),
    (30000, 8, 1, True, "bf16", "ties"),
    (20000, 64, 6, False, "bf16", "extremes"),
    (20000, 32, 5, True, "f16", "extremes"),
    # E = 64: TMA-fed tiles of 128 rows, several tiles per CTA through the
    # slot ring at the larger T, one ragged tile at the smallest
    (9729, 64, 1, False, "f16", "specials"),
    (40000, 64, 7, True, "f16", "extremes"),
    (400000, 64, 8, True, "f16", "ties"),
    (700001, 64, 6, False, "bf16", "normal"),
]


def _route_logits(T, E, ldt, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "ties":
        l = torch.randint(-2, 3, (T, E), generator=g).float() * 0.5
    else:
        l = torch.randn((T, E), generator=g)
    if kind == "extremes":
        # rows near the dtype's largest values (BF16 ~3.4e38: exp(l - m) of
        # such rows; F16 turns them into +-inf rows) and rows of subnormals
        # (BF16 keeps 1e-39-scale values and their order; F16 makes them 0)
        l[0::4] *= 1.0e38
        l[1::4] *= 1.0e-39
        l[2::4, ::2] *= 1.0e38
        l[2::4, 1::2] *= 1.0e-39
    if kind == "specials":
        l[0, 3] = float("nan")
        l[1, :] = float("-inf")
        l[2, 5] = float("inf")
        l[3, ::2] = float("-inf")           # valid: finite and -inf mixed
        l[4, :] = float("-inf")
        l[4, E - 1] = 0.0                    # one finite entry, k > 1
        l[5, 0] = float("-inf")
        l[5, 1] = float("inf")
        l[6, :] = 0.0                        # all tied
        l[7, :] = -0.0
        l[7, 2] = 0.0                        # +0 and -0 tie
    return l.to(W.TORCH_DTYPES[ldt])


@pytest.mark.parametrize("T,E,k,renorm,ldt,kind", ROUTE_CASES)
def test_route_parity(dev, T, E, k, renorm, ldt, kind):
    logits = _route_logits(T, E, ldt, kind, seed=T * 131 + E)
    idx_ref, w_ref, _ = oracle.route(np_of(logits), ldt, k, renorm)
    idx, w = moe.moe_route(logits.to(dev), k, renorm)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy().view(np.uint32), idx_ref), "expert ids differ"
    assert_close(to_f64(w), oracle.to_f64(w_ref, ldt), ldt if ldt != "f32" else "f32", "weights")


def test_route_workload_logits(dev):
    for cfg in list(W.CONFIGS.values()):
        logits = W.moe_inputs(cfg.scaled(I=8, H=8), device="cpu")["logits"]
        idx_ref, w_ref, inval = oracle.route(np_of(logits), cfg.logits_dtype, cfg.top_k,
                                             cfg.renormalize)
        idx, w = moe.moe_route(logits.to(dev), cfg.top_k, cfg.renormalize)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy().view(np.uint32), idx_ref), cfg.name
        assert_close(to_f64(w), oracle.to_f64(w_ref, cfg.logits_dtype), cfg.logits_dtype,
                     cfg.name)
    cn = W.COMBINE_NORM
    logits = W.combine_norm_inputs(cn.scaled(T=cn.T, H=8), device="cpu")["logits"]
    idx_ref, w_ref, _ = oracle.route(np_of(logits), "f32", cn.top_k, True)
    idx, w = moe.moe_route(logits.to(dev), cn.top_k, True)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy().view(np.uint32), idx_ref)
    assert_close(to_f64(w), w_ref.astype(np.float64), "f32", "combine-norm routing")


def test_route_empty(dev):
    idx, w = moe.moe_route(torch.empty((0, 8), device=dev), 2, True)
    assert idx.shape == (0, 2) and w.shape == (0, 2)


# ---------------------------------------------------------------- dispatch

def _check_dispatch(d, idx_np, x_np, E, k, dt):
    counts, offsets, row_of, src_of, bad = oracle.dispatch(idx_np, E)
    g_counts = d["counts"].cpu().numpy()
    g_offsets = d["offsets"].cpu().numpy()
    g_row = d["row_of"].cpu().numpy()
    g_src = d["src_of"].cpu().numpy()
    assert np.array_equal(g_counts, counts) and np.array_equal(g_offsets, offsets)
    rows = int(offsets[E])
    assert per_expert_sets(g_src[:rows], offsets) == per_expert_sets(src_of[:rows], offsets)
    valid = row_of >= 0
    assert np.array_equal(g_row < 0, ~valid)
    assert np.array_equal(g_src[g_row[valid]], np.nonzero(valid)[0])
    # this implementation is stable: rows follow the assignment order
    assert np.array_equal(g_row, row_of) and np.array_equal(g_src[:rows], src_of[:rows])
    xd = np_of(d["x_disp"])[:rows]
    assert np.array_equal(xd, oracle.gather(x_np, dt, k, src_of, rows))


DISPATCH_CASES = [(4096, 6, 64, 2048, "bf16"), (8192, 8, 256, 64, "bf16"),
                  (16384, 2, 8, 64, "f32"), (128, 8, 256, 7168, "bf16"),
                  (37, 3, 5, 24, "f16"), (1, 1, 1, 8, "f32"), (500, 4, 1024, 8, "bf16"),
                  (3000, 1, 4, 40, "bf16"),
                  # x past 32 MiB with rows of >= 512 bytes: the token-order gather
                  # (k = 40 reads the slots' rows in two groups of 32 lanes)
                  (9000, 3, 16, 2048, "bf16"), (5000, 40, 64, 1792, "f32"),
                  (8200, 2, 8, 4096, "f16"),
                  # rank counters in registers (E <= 64: experts lane and lane + 32)
                  # around their edges, and E = 100 (seven key bits, shared memory)
                  (20000, 6, 33, 8, "bf16"), (30000, 8, 64, 16, "f16"),
                  (5000, 5, 32, 8, "f32"), (20000, 4, 100, 8, "bf16")]


@pytest.mark.parametrize("T,k,E,H,dt", DISPATCH_CASES)
def test_dispatch_parity(dev, T, k, E, H, dt):
    g = torch.Generator().manual_seed(T + k * 7 + E)
    if E > 1 and T == 3000:
        idx = torch.zeros((T, k), dtype=torch.int32)          # every token to expert 0
    else:
        idx = torch.stack([torch.randperm(E, generator=g)[:k] if k <= E else
                           torch.randint(0, E, (k,), generator=g) for _ in range(T)]).int()
    x = (torch.randn((T, H), generator=g)).to(W.TORCH_DTYPES[dt])
    d = moe.moe_dispatch(idx.to(dev), x.to(dev), E)
    torch.cuda.synchronize()
    _check_dispatch(d, idx.numpy().view(np.uint32), np_of(x), E, k, dt)
    assert moe.moe_device_status() == 0


@pytest.mark.parametrize("E", [33, 64, 100])
def test_dispatch_bad_indices_many_experts(dev, E):
    """Ids >= E among many experts get no row and are flagged; the rows of the
    others stay bit-exact (rank counters in registers up to 64 experts)."""
    T, k, H = 20000, 4, 8
    g = torch.Generator().manual_seed(E)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).int()
    bad = torch.randint(0, T, (50,), generator=g)
    idx[bad, 1] = E + torch.randint(0, 1000, (50,), generator=g).int()
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    assert moe.moe_device_status(clear=True) == 0
    d = moe.moe_dispatch(idx.to(dev), x.to(dev), E)
    assert moe.moe_device_status(clear=True) == 9        # MOE_ERR_BAD_INDEX
    _check_dispatch(d, idx.numpy().view(np.uint32), np_of(x), E, k, "bf16")


def test_dispatch_bad_index_flags_and_nans(dev):
    T, k, E, H = 40, 2, 4, 16
    g = torch.Generator().manual_seed(5)
    idx = torch.randint(0, E, (T, k), generator=g).int()
    idx[3, 1] = 7
    idx[10, 0] = 2 ** 31 - 1
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    assert moe.moe_device_status(clear=True) == 0
    d = moe.moe_dispatch(idx.to(dev), x.to(dev), E)
    assert moe.moe_device_status(clear=True) == 9        # MOE_ERR_BAD_INDEX
    assert moe.moe_device_status(clear=True) == 0        # cleared
    _check_dispatch(d, idx.numpy().view(np.uint32), np_of(x), E, k, "bf16")
    w = torch.full((T, k), 0.5, device=dev)
    out = torch.randn((T * k, H), device=dev).to(torch.bfloat16)
    y = moe.moe_combine(out, w, d["row_of"])
    torch.cuda.synchronize()
    nan_rows = torch.isnan(y.float()).all(dim=1).cpu().numpy()
    assert nan_rows[3] and nan_rows[10] and nan_rows.sum() == 2


# ---------------------------------------------------------------- experts

@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
@pytest.mark.parametrize("out_f32", [False, True], ids=["out_dtype", "out_f32"])
def test_experts_parity(dev, cfg, out_f32):
    if out_f32 and cfg.dtype == "f32":
        pytest.skip("FP32 experts always write FP32")
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    idx, _, _ = oracle.route(o["logits"], cfg.logits_dtype, cfg.top_k, cfg.renormalize)
    _, offsets, _, src_of, _ = oracle.dispatch(idx, cfg.E)
    rows = int(offsets[cfg.E])
    x_disp = oracle.gather(o["x"], cfg.dtype, cfg.top_k, src_of, rows)
    ref = oracle.experts_dispatched(x_disp, cfg.dtype, offsets, o["gate"], o["up"], o["down"])
    xd = W.from_numpy(x_disp, cfg.dtype, dev)
    out = moe.moe_experts_forward(xd, torch.from_numpy(offsets).to(dev), g["gate"],
                                  g["up"], g["down"],
                                  out_dtype=torch.float32 if out_f32 else None)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    # FP32 outputs of BF16/F16 experts still carry the rounding of h to the
    # input dtype between the GEMMs, so they are held to the input dtype's bar
    assert_close(to_f64(out), ref, cfg.dtype, f"{cfg.name} expert outputs")


@pytest.mark.parametrize("cfg", [SMALL[0], PAIR[0]], ids=lambda c: c.name)
def test_experts_rows_beyond_offsets_untouched(dev, cfg):
    """offsets[E] < rows: rows past the last segment are not written."""
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    idx, _, _ = oracle.route(o["logits"], cfg.logits_dtype, cfg.top_k, cfg.renormalize)
    _, offsets, _, src_of, _ = oracle.dispatch(idx, cfg.E)
    rows = int(offsets[cfg.E])
    x_disp = oracle.gather(o["x"], cfg.dtype, cfg.top_k, src_of, rows)
    pad = np.zeros((rows + 77, cfg.H), np.uint16)
    pad[:rows] = x_disp
    xd = W.from_numpy(pad, cfg.dtype, dev)
    out = torch.full((rows + 77, cfg.H), 3.0, dtype=torch.bfloat16, device=dev)
    moe.moe_experts_forward(xd, torch.from_numpy(offsets).to(dev), g["gate"], g["up"],
                            g["down"], out_disp=out)
    torch.cuda.synchronize()
    assert torch.all(out[rows:].float() == 3.0)
    ref = oracle.experts_dispatched(x_disp, cfg.dtype, offsets, o["gate"], o["up"], o["down"])
    assert_close(to_f64(out[:rows]), ref, cfg.dtype, "prefix rows")


@pytest.mark.parametrize("T,split", [(200, 50), (800, 300)], ids=["single", "pair"])
def test_experts_exact_small_integers(dev, T, split):
    """Integer-valued BF16 inputs with gate = 0 rows make SiLU exact (h = 0
    where g = 0); up/down chosen so every product and FP32 sum is exact.
    Expert 1 is empty; T = 800 (>= 2 x 128 rows per expert) runs CTA pairs."""
    E, I, H = 3, 128, 64
    g = torch.Generator().manual_seed(3)
    x = torch.randint(-3, 4, (T, H), generator=g).to(torch.bfloat16)
    gate = torch.zeros((E, I, H), dtype=torch.bfloat16)
    up = torch.randint(-2, 3, (E, I, H), generator=g).to(torch.bfloat16)
    down = torch.randint(-2, 3, (E, H, I), generator=g).to(torch.bfloat16)
    offsets = torch.tensor([0, split, split, T], dtype=torch.int32)
    out = moe.moe_experts_forward(x.to(dev), offsets.to(dev), gate.to(dev), up.to(dev),
                                  down.to(dev))
    torch.cuda.synchronize()
    assert torch.all(out.cpu().float() == 0.0)


# Rows per expert around the edges of the CTA-pair units (256 rows each; an
# expert's last unit with at most 128 rows runs as an M = 128 pair tile, 64
# rows per CTA): one full unit (256), exactly one M = 128 tile (128), a single
# row (1), one CTA's rows only (64) and one more (65), a full unit with one row
# on its second CTA (129), 383 / 384 / 385 around the fine prefill's average,
# an empty expert, and a long one. 3095 rows >= 256 per expert select pairs;
# H = 200 leaves a K tail, I = 200 partial N tiles in both GEMMs.
PAIR_EDGE_COUNTS = [256, 128, 1, 64, 65, 129, 383, 384, 385, 0, 200, 1100]


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_experts_pair_unit_edges(dev, dt):
    E, H, I = len(PAIR_EDGE_COUNTS), 200, 200
    offsets = np.concatenate([[0], np.cumsum(PAIR_EDGE_COUNTS)]).astype(np.int32)
    rows = int(offsets[-1])
    assert rows >= 256 * E
    g = torch.Generator().manual_seed(11)
    x = torch.randn((rows, H), generator=g).to(dt)
    gate = (torch.randn((E, I, H), generator=g) * H ** -0.5).to(dt)
    up = (torch.randn((E, I, H), generator=g) * H ** -0.5).to(dt)
    down = (torch.randn((E, H, I), generator=g) * I ** -0.5).to(dt)
    name = TORCH_TO_NAME[dt]
    off = torch.from_numpy(offsets).to(dev)
    on = [t.to(dev) for t in (x, gate, up, down)]
    out16 = moe.moe_experts_forward(*on[:1], off, *on[1:])
    out32 = moe.moe_experts_forward(*on[:1], off, *on[1:], out_dtype=torch.float32)
    out_t, cache = moe.moe_experts_forward_training(*on[:1], off, *on[1:],
                                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.experts_dispatched(np_of(x), name, offsets, np_of(gate), np_of(up), np_of(down))
    assert_close(to_f64(out16), ref, name, "expert outputs (dtype)")
    assert_close(to_f64(out32), ref, name, "expert outputs (FP32)")
    assert torch.equal(out_t, out32)
    hb = rows * I * x.element_size()
    h_c = cache[:hb].view(dt).view(rows, I)
    gu_c = cache[hb: hb + 2 * rows * I * 4].view(torch.float32).view(2, rows, I)
    rg, ru, rh = oracle.experts_cache_dispatched(np_of(x), name, offsets, np_of(gate), np_of(up))
    assert_close(to_f64(gu_c[0]), rg, name, "cached g")
    assert_close(to_f64(gu_c[1]), ru, name, "cached u")
    assert_close(to_f64(h_c), rh, name, "cached h")


# Experts averaging >= 2048 rows run their CTA pairs with two k-blocks per
# pipeline stage. Counts: 8 full units + a unit with one row on its second
# CTA (2177), 15 full units + an M = 128 tile of 60 rows (3900), exactly one
# M = 128 tile (128). (H, I) = (192, 320): odd k-block counts, two-k-block
# boxes with the second k-block past K in each unit's last stage;
# (200, 136): K tails, so one box per k-block in two-k-block stages.
TWO_KB_COUNTS = [2177, 3900, 128]


@pytest.mark.parametrize("H,I", [(192, 320), (200, 136)], ids=["boxes", "k_tails"])
def test_experts_two_kblock_stages(dev, H, I):
    dt = torch.bfloat16
    E = len(TWO_KB_COUNTS)
    offsets = np.concatenate([[0], np.cumsum(TWO_KB_COUNTS)]).astype(np.int32)
    rows = int(offsets[-1])
    assert rows >= 2048 * E
    g = torch.Generator().manual_seed(13)
    x = torch.randn((rows, H), generator=g).to(dt)
    gate = (torch.randn((E, I, H), generator=g) * H ** -0.5).to(dt)
    up = (torch.randn((E, I, H), generator=g) * H ** -0.5).to(dt)
    down = (torch.randn((E, H, I), generator=g) * I ** -0.5).to(dt)
    off = torch.from_numpy(offsets).to(dev)
    on = [t.to(dev) for t in (x, gate, up, down)]
    out16 = moe.moe_experts_forward(*on[:1], off, *on[1:])
    out_t, cache = moe.moe_experts_forward_training(*on[:1], off, *on[1:],
                                                    out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    ref = oracle.experts_dispatched(np_of(x), "bf16", offsets, np_of(gate), np_of(up),
                                    np_of(down))
    assert_close(to_f64(out16), ref, "bf16", "expert outputs (dtype)")
    assert_close(to_f64(out_t), ref, "bf16", "expert outputs (FP32, training)")
    hb = rows * I * 2
    h_c = cache[:hb].view(dt).view(rows, I)
    gu_c = cache[hb: hb + 2 * rows * I * 4].view(torch.float32).view(2, rows, I)
    rg, ru, rh = oracle.experts_cache_dispatched(np_of(x), "bf16", offsets, np_of(gate),
                                                 np_of(up))
    assert_close(to_f64(gu_c[0]), rg, "bf16", "cached g")
    assert_close(to_f64(gu_c[1]), ru, "bf16", "cached u")
    assert_close(to_f64(h_c), rh, "bf16", "cached h")


# ---------------------------------------------------------------- combine

# (T, k, H, expert-output dtype, weight dtype, activation dtype)
COMBINE_CASES = [(300, 2, 320, "bf16", "f32", "bf16"), (4096, 6, 2048, "bf16", "bf16", "bf16"),
                 (64, 2, 128, "f32", "f32", "f32"), (129, 8, 7168, "bf16", "f32", "bf16"),
                 (77, 3, 264, "f16", "f16", "f16"), (5, 1, 16384, "bf16", "f32", "bf16"),
                 (300, 6, 2048, "f32", "bf16", "bf16"), (90, 4, 520, "f32", "f32", "f16")]


def _routing_for(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn((T, E), generator=g)
    logits[1 % T, 0] = float("nan")
    idx, w, _ = oracle.route(logits.numpy(), "f32", k, True)
    _, _, row_of, _, _ = oracle.dispatch(idx, E)
    return w, row_of


@pytest.mark.parametrize("T,k,H,odt,wdt,dt", COMBINE_CASES)
def test_combine_parity(dev, T, k, H, odt, wdt, dt):
    E = max(k, 16)
    w, row_of = _routing_for(T, k, E, seed=T + H)
    wt = torch.from_numpy(w)
    if wdt != "f32":
        wt = wt.to(W.TORCH_DTYPES[wdt])
    g = torch.Generator().manual_seed(H)
    out = torch.randn((T * k, H), generator=g).to(W.TORCH_DTYPES[odt])
    ref = oracle.combine(np_of(out), odt, np_of(wt), wdt, row_of, k)
    y = moe.moe_combine(out.to(dev), wt.to(dev), torch.from_numpy(row_of).to(dev),
                        dtype=W.TORCH_DTYPES[dt])
    torch.cuda.synchronize()
    assert y.dtype == W.TORCH_DTYPES[dt]
    assert_close(to_f64(y), ref, dt, "combine")


@pytest.mark.parametrize("T,k,H,odt,wdt,dt", COMBINE_CASES)
@pytest.mark.parametrize("gdt", ["same", "f32"])
def test_combine_add_rmsnorm_parity(dev, T, k, H, odt, wdt, dt, gdt):
    E = max(k, 16)
    w, row_of = _routing_for(T, k, E, seed=T * 3 + H)
    wt = torch.from_numpy(w)
    if wdt != "f32":
        wt = wt.to(W.TORCH_DTYPES[wdt])
    g = torch.Generator().manual_seed(H + 1)
    tdt = W.TORCH_DTYPES[dt]
    out = torch.randn((T * k, H), generator=g).to(W.TORCH_DTYPES[odt])
    res = torch.randn((T, H), generator=g).to(tdt)
    gdt_name = dt if gdt == "same" else "f32"
    gamma = (1 + math.sqrt(0.1) * torch.randn(H, generator=g)).to(W.TORCH_DTYPES[gdt_name])
    eps = 1e-6
    comb = oracle.combine(np_of(out), odt, np_of(wt), wdt, row_of, k)
    y_ref, x_ref, rstd_ref = oracle.add_rmsnorm(comb, np_of(res), dt, np_of(gamma),
                                                gdt_name, eps)
    y, x_out, rstd = moe.moe_combine_add_rmsnorm(
        out.to(dev), wt.to(dev), torch.from_numpy(row_of).to(dev), res.to(dev),
        gamma.to(dev), eps)
    torch.cuda.synchronize()
    assert_close(to_f64(x_out), oracle.to_f64(x_ref, dt), dt, "x_out")
    assert_close(to_f64(y), oracle.to_f64(y_ref, dt), dt, "y")
    assert_close(rstd.cpu().numpy().astype(np.float64), rstd_ref.astype(np.float64),
                 "f32", "rstd")


def test_combine_one_hot_is_exact_gather(dev):
    T, k, H = 100, 4, 256
    g = torch.Generator().manual_seed(9)
    out = torch.randn((T * k, H), generator=g).to(torch.bfloat16)
    row_of = torch.randperm(T * k, generator=g).int()
    pick = torch.randint(0, k, (T,), generator=g)
    w = torch.zeros((T, k))
    w[torch.arange(T), pick] = 1.0
    y = moe.moe_combine(out.to(dev), w.to(dev), row_of.to(dev)).cpu()
    want = out[row_of.view(T, k)[torch.arange(T), pick].long()]
    assert torch.equal(y, want)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_forward_parity(dev, cfg):
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"],
                         o["up"], o["down"], cfg.top_k, cfg.renormalize)
    y = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                        cfg.renormalize)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert_close(to_f64(y), ref["y"], cfg.dtype, f"{cfg.name} y")
    # the staged calls compute the same thing; for FP32 through the same
    # kernels (bit for bit), for BF16/F16 with the combine as a separate,
    # deterministic kernel instead of reductions inside the second GEMM
    idx, w = moe.moe_route(g["logits"], cfg.top_k, cfg.renormalize)
    d = moe.moe_dispatch(idx, g["x"], cfg.E)
    out = moe.moe_experts_forward(d["x_disp"], d["offsets"], g["gate"], g["up"], g["down"],
                                  out_dtype=torch.float32)
    y2 = moe.moe_combine(out, w, d["row_of"], dtype=g["x"].dtype)
    torch.cuda.synchronize()
    assert torch.equal(torch.isnan(y), torch.isnan(y2))
    if cfg.dtype == "f32":
        assert torch.equal(torch.nan_to_num(y), torch.nan_to_num(y2))
    else:
        assert_close(to_f64(y2), ref["y"], cfg.dtype, f"{cfg.name} staged y")
        assert_same_sum(y, y2, combine_magnitude(out, w, d["row_of"]), cfg.top_k)


def test_forward_tiny_fp32_special_rows(dev):
    cfg = W.CONFIGS["tiny_fp32"]
    cpu, g = inputs_on(cfg, dev)
    y = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], 2, True).cpu()
    nan_rows = torch.isnan(y).all(dim=1)
    assert nan_rows[4] and nan_rows[5] and int(nan_rows.sum()) == 2


def combine_magnitude(out: torch.Tensor, w: torch.Tensor, row_of: torch.Tensor) -> torch.Tensor:
    """sum_j |w[t,j]| * |o[row_of[t,j]]| per output element (FP32)."""
    return moe.moe_combine(out.abs(), w.float().abs(), row_of, dtype=torch.float32)


def assert_same_sum(a: torch.Tensor, b: torch.Tensor, mag: torch.Tensor, k: int):
    """Two outputs of the same k-term FP32 sums of products w*o, formed with
    different roundings and orders (separate products and reductions in
    arrival order, or fused multiply-adds in slot order): equal NaN rows, and
    apart by at most the two FP32 sums' error bound, k * 2^-23 * sum|w*o|
    (each side within k * 2^-24 * sum|w*o| of the exact sum), plus one unit in
    the last place of the output dtype for the final roundings."""
    assert torch.equal(torch.isnan(a), torch.isnan(b))
    fa, fb = torch.nan_to_num(a.float()), torch.nan_to_num(b.float())
    mant = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}[a.dtype]
    big = torch.maximum(fa.abs(), fb.abs()).clamp_min(1e-30)
    ulp = torch.exp2(torch.floor(torch.log2(big)) - mant)
    bound = ulp + k * 2.0 ** -23 * torch.nan_to_num(mag)
    assert torch.all((fa - fb).abs() <= bound), float(((fa - fb).abs() / bound).max())


def test_forward_repeatable_and_stream(dev):
    cfg = SMALL[1]
    _, g = inputs_on(cfg, dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"],
                             cfg.top_k, cfg.renormalize, stream=s)
        y2 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"],
                             cfg.top_k, cfg.renormalize, stream=s)
    s.synchronize()
    # the staged path is bit-reproducible
    idx, w = moe.moe_route(g["logits"], cfg.top_k, cfg.renormalize)
    d = moe.moe_dispatch(idx, g["x"], cfg.E)
    ys = []
    for _ in range(2):
        out = moe.moe_experts_forward(d["x_disp"], d["offsets"], g["gate"], g["up"],
                                      g["down"], out_dtype=torch.float32)
        ys.append(moe.moe_combine(out, w, d["row_of"], dtype=g["x"].dtype))
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1])
    # the one-call forward's reductions arrive in any order
    assert_same_sum(y1, y2, combine_magnitude(out, w, d["row_of"]), cfg.top_k)


# The one-call forward's fused routing-and-count kernel on every width it is
# compiled for (lanes per token 16 / 32, logits per lane 8 / 16 / 32), with
# dispatch chunks of 256 assignments whose edges split tokens (top_k 3, 6, 7).
FUSED_FRONT = [
    cfg_small("fused_e100_bf16", T=300, H=64, I=64, E=100, top_k=3, renormalize=True,
              dtype="bf16", logits_dtype="bf16"),
    cfg_small("fused_e300_bf16", T=200, H=64, I=32, E=300, top_k=7, renormalize=False,
              dtype="bf16", logits_dtype="f32", logit_bias="zipf", bias_param=1.1),
    cfg_small("fused_e700_f16", T=150, H=32, I=32, E=700, top_k=6, renormalize=True,
              dtype="f16", logits_dtype="f16"),
    cfg_small("fused_e1024_bf16", T=120, H=32, I=32, E=1024, top_k=8, renormalize=True,
              dtype="bf16", logits_dtype="bf16"),
]


# The smallest batches: one token, and three tokens over 16 experts (one
# dispatch chunk; most experts get no rows, so GEMM2 starts on few experts).
TINY_BATCH = [
    cfg_small("one_token_bf16", T=1, H=64, I=64, E=4, top_k=2, renormalize=True,
              dtype="bf16", logits_dtype="bf16"),
    cfg_small("three_tokens_f16", T=3, H=128, I=96, E=16, top_k=4, renormalize=False,
              dtype="f16", logits_dtype="f32"),
]


@pytest.mark.parametrize("cfg", TINY_BATCH, ids=lambda c: c.name)
def test_forward_tiny_batches(dev, cfg):
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"],
                         o["up"], o["down"], cfg.top_k, cfg.renormalize)
    y = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                        cfg.renormalize)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert_close(to_f64(y), ref["y"], cfg.dtype, f"{cfg.name} y")


@pytest.mark.parametrize("cfg", FUSED_FRONT, ids=lambda c: c.name)
def test_forward_fused_front_wide_experts(dev, cfg):
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    ref = oracle.forward(o["x"], cfg.dtype, o["logits"], cfg.logits_dtype, o["gate"],
                         o["up"], o["down"], cfg.top_k, cfg.renormalize)
    y = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                        cfg.renormalize)
    torch.cuda.synchronize()
    assert moe.moe_device_status() == 0
    assert_close(to_f64(y), ref["y"], cfg.dtype, f"{cfg.name} y")
    # the standalone routing computes the ids the forward used
    idx, _ = moe.moe_route(g["logits"], cfg.top_k, cfg.renormalize)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy().astype(np.uint32), ref["idx"])


@pytest.mark.parametrize("cfg", [SMALL[0], PAIR[0]], ids=lambda c: c.name)
def test_forward_cuda_graph_replay(dev, cfg):
    """moe_forward captured once in a CUDA graph (its workspace memset, the
    routing, dispatch, GEMM and finalize kernels, their programmatic-launch
    edges) computes the forward of whatever the captured input buffers hold
    at each replay."""
    cpu, g = inputs_on(cfg, dev)
    o = oracle_inputs(cpu)
    x, logits = g["x"].clone(), g["logits"].clone()
    ws = torch.empty(moe.moe_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k,
                                                    x.dtype, logits.dtype),
                     dtype=torch.uint8, device=dev)
    y = torch.empty_like(x)

    def fwd():
        moe.moe_forward(x, logits, g["gate"], g["up"], g["down"], cfg.top_k, cfg.renormalize,
                        y=y, workspace=ws)

    fwd()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for seed in (5, 6):
        gen = torch.Generator().manual_seed(seed)
        x.copy_(torch.randn(x.shape, generator=gen).to(x.dtype))
        logits.copy_(torch.randn(logits.shape, generator=gen).to(logits.dtype))
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_device_status() == 0
        ref = oracle.forward(np_of(x), cfg.dtype, np_of(logits), cfg.logits_dtype, o["gate"],
                             o["up"], o["down"], cfg.top_k, cfg.renormalize)
        assert_close(to_f64(y), ref["y"], cfg.dtype, f"{cfg.name} y, graph replay {seed}")


def test_forward_fp32_bit_reproducible(dev):
    cfg = SMALL[5]
    _, g = inputs_on(cfg, dev)
    y1 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                         cfg.renormalize)
    y2 = moe.moe_forward(g["x"], g["logits"], g["gate"], g["up"], g["down"], cfg.top_k,
                         cfg.renormalize)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_forward_empty_batch(dev):
    cfg = SMALL[0]
    _, g = inputs_on(cfg, dev)
    y = moe.moe_forward(g["x"][:0], g["logits"][:0], g["gate"], g["up"], g["down"],
                        cfg.top_k, cfg.renormalize)
    assert y.shape == (0, cfg.H)
