"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each ``check_*`` takes a loaded oracle library (the real one, or a
deliberately broken build in ``test_oracle_mutants.py``) and raises
``AssertionError`` when the oracle disagrees with:

* hand-derived closed forms of the routing, SwiGLU and RMSNorm rules
  (``tests/golden/``);
* library routines the rules reduce to (``scipy.special.softmax`` when
  top_k = E, numpy's sort for the selection, numpy matmul for a dense
  evaluation of the experts, torch / numpy dtype casts);
* invariants: permutation bijections, weight sums, linearity, exact integer
  arithmetic.

Sources: ruDNN user guide sections 3-7; aclnnMoeDistributeCombineAddRmsNormV2
"Function" formula; aclnnFFN "Formula".
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


_EXPR_NS = {"sig": _sig, "exp": math.exp, "sqrt": math.sqrt, "nan": math.nan,
            "inf": math.inf, "__builtins__": {}}


def _eval(expr: str, **extra) -> float:
    ns = dict(_EXPR_NS)
    ns.update(extra)
    return float(eval(expr, ns))  # fixtures are repository text


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


def _logit(tok: str) -> float:
    if tok.startswith("ln:"):
        return math.log(float(tok[3:]))
    return float(tok)


def _f32_close(a, b, rel=4e-7):
    return abs(a - b) <= rel * max(abs(a), abs(b), 1e-30) + 1e-37


# ---------------------------------------------------------------- conversions

def check_conversions(lib):
    """bf16 RNE against torch's cast, f16 against numpy's, exact upcasts."""
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        rng.standard_normal(1000).astype(np.float32) * 1e-38,
        np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 65504.0, 70000.0,
                  3.0e38, 1.00390625, 1.01171875, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8],
                 dtype=np.float32)])
    bf = oracle.convert(vals, "f32", "bf16", lib)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, ref), "bf16 rounding differs from torch"
    back = oracle.convert(bf, "bf16", "f32", lib)
    ref_back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(back, ref_back), "bf16 upcast not exact"
    h = oracle.convert(vals, "f32", "f16", lib)
    with np.errstate(over="ignore"):
        ref16 = vals.astype(np.float16)
    assert np.array_equal(h, ref16.view(np.uint16)), "f16 rounding"
    hb = oracle.convert(h, "f16", "f32", lib)
    assert np.array_equal(hb, h.view(np.float16).astype(np.float32)), "f16 upcast"
    nan_bf = oracle.convert(np.array([np.nan], np.float32), "f32", "bf16", lib)
    assert np.isnan(oracle.convert(nan_bf, "bf16", "f32", lib)[0])


# -------------------------------------------------------------------- routing

def check_route_golden(lib):
    """Hand-derived routing cases (ruDNN user guide, section 4)."""
    n = 0
    for fields in _lines("routing_cases.txt"):
        E, k, ren = (int(v) for v in fields[0].split())
        logits = np.array([[_logit(v) for v in fields[1].split()]], np.float32)
        want_idx = [int(v) for v in fields[2].split()]
        want_w = fields[3].split()
        idx, w, _ = oracle.route(logits, "f32", k, bool(ren), lib)
        assert list(idx[0]) == want_idx, (fields, idx)
        for got, want in zip(w[0], want_w):
            if want == ".":
                continue
            if want == "nan":
                assert math.isnan(got), (fields, w)
            else:
                assert _f32_close(float(got), float(Fraction(want))), (fields, w)
        n += 1
    assert n >= 10


def check_route_planted_rows(lib):
    """The tiny FP32 workload plants ties, a NaN row and an all -inf row
    (rows 0-5); their routing is fixed by the routing rules alone."""
    from mixture_experts_ffn_topk_gb300 import workloads as W
    cfg = W.CONFIGS["tiny_fp32"]
    logits = W.to_numpy(W.moe_inputs(cfg)["logits"])
    idx, w, invalid = oracle.route(logits, "f32", 2, True, lib)
    assert idx[:6].tolist() == [[2, 6], [1, 4], [7, 3], [0, 2], [0, 1], [0, 1]]
    assert w[0].tolist() == [0.5, 0.5] and w[1].tolist() == [0.5, 0.5]
    assert np.isnan(w[4]).all() and np.isnan(w[5]).all()
    assert invalid == 2
    # rows 2 and 3: top logit 5, runner-up 4 -> renormalised weights are
    # sig(1) and 1 - sig(1)
    for r in (2, 3):
        assert _f32_close(float(w[r, 0]), _sig(1.0), 2e-7)
        assert _f32_close(float(w[r, 1]), 1.0 - _sig(1.0), 2e-6)


def check_route_full_softmax(lib):
    """top_k = E returns the whole softmax (a library routine) in descending
    order; with renormalisation the weights are unchanged up to rounding."""
    rng = np.random.default_rng(11)
    for E in (1, 2, 3, 8, 33, 64, 257):
        logits = (rng.standard_normal((9, E)) * 3).astype(np.float32)
        ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
        for ren in (False, True):
            idx, w, _ = oracle.route(logits, "f32", E, ren, lib)
            for t in range(9):
                assert sorted(idx[t].tolist()) == list(range(E))
                np.testing.assert_allclose(w[t], ref[t, idx[t]], rtol=3e-6,
                                           atol=1e-12)
                assert np.all(np.diff(ref[t, idx[t]]) <= 1e-12)


def _sg_case(fields):
    E, G, S, k, two, ren = (int(v) for v in fields[0].split()[:6])
    scale = float(Fraction(fields[0].split()[6]))
    def tok(v):
        return -_logit(v[1:]) if v.startswith("-ln:") else _logit(v)
    logits = np.array([[tok(v) for v in fields[1].split()]], np.float32)
    bias = None if fields[2] == "none" else np.array(
        [float(Fraction(v)) if v != "nan" else math.nan for v in fields[2].split()], np.float32)
    return E, G, S, k, two, ren, scale, logits, bias


def check_sigmoid_grouped_golden(lib):
    """Hand-derived group-limited sigmoid routing cases (ruDNN user guide,
    section 10)."""
    n = 0
    for fields in _lines("sigmoid_grouped_cases.txt"):
        E, G, S, k, two, ren, scale, logits, bias = _sg_case(fields)
        assert logits.shape == (1, E)
        idx, w, _ = oracle.route_sigmoid_grouped(logits, "f32", bias, k, G, S, bool(two),
                                                 bool(ren), scale, lib)
        want_idx = [int(v) for v in fields[3].split()]
        assert list(idx[0]) == want_idx, (fields, idx)
        for got, want in zip(w[0], fields[4].split()):
            if want == "nan":
                assert math.isnan(got), (fields, w)
            else:
                assert _f32_close(float(got), float(Fraction(want)), 1e-6), (fields, w)
        n += 1
    assert n >= 12


def _group_scores(c, G, two):
    per = np.sort(c.reshape(G, -1), axis=1)[:, ::-1]
    return per[:, 0] + per[:, 1] if two else per[:, 0]


def check_sigmoid_grouped_optimality(lib):
    """Random rows against the selection rule stated as order conditions
    (checked with sorts, not the oracle's scans): every kept group ranks
    before every dropped one on (score desc, id asc); the picked experts lie
    in kept groups and rank before every unpicked expert of those groups on
    (corrected score desc, id asc), in pick order; weights are the closed-form
    sigmoid of the picked logits, renormalised and scaled."""
    rng = np.random.default_rng(41)
    for trial in range(60):
        G = int(rng.choice([1, 2, 4, 8]))
        gs = int(rng.choice([2, 3, 4]))
        E = G * gs
        S = int(rng.integers(1, G + 1))
        k = int(rng.integers(1, S * gs + 1))
        two, ren = bool(trial % 2), bool(trial % 3 == 0)
        scale = float(rng.choice([1.0, 2.5]))
        T = 7
        logits = np.round(rng.standard_normal((T, E)) * 2, 1).astype(np.float32)  # ties happen
        bias = (np.round(rng.standard_normal(E), 1) * 0.2).astype(np.float32) if trial % 4 else None
        idx, w, bad = oracle.route_sigmoid_grouped(logits, "f32", bias, k, G, S, two, ren,
                                                   scale, lib)
        assert bad == 0
        for t in range(T):
            s = (1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)))).astype(np.float32)
            c = s + (bias if bias is not None else np.float32(0))
            gsc = _group_scores(c, G, two)
            order_g = np.lexsort((np.arange(G), -gsc.astype(np.float64)))
            kept = set(order_g[:S].tolist())
            cand = [e for e in range(E) if e // gs in kept]
            order_e = sorted(cand, key=lambda e: (-float(c[e]), e))
            assert idx[t].tolist() == order_e[:k], (trial, t)
            sel = s[idx[t]].astype(np.float64)
            if ren:
                sel = sel / sel.sum()
            assert np.allclose(w[t], sel * scale, rtol=2e-6, atol=0), (trial, t)


def check_sigmoid_grouped_reduces_to_softmax_order(lib):
    """One group, no bias: sigmoid is increasing, so the picks are the top-k
    logits -- the same ids as the (separately pinned) softmax routing, for
    logits far from sigmoid saturation."""
    rng = np.random.default_rng(43)
    logits = (rng.standard_normal((50, 40)) * 2).astype(np.float32)
    for k in (1, 5, 40):
        ids, _, _ = oracle.route_sigmoid_grouped(logits, "f32", None, k, 1, 1, False, False,
                                                 1.0, lib)
        ref, _, _ = oracle.route(logits, "f32", k, False, lib)
        assert np.array_equal(ids, ref)


def check_sigmoid_grouped_arguments(lib):
    """Limits the section states are rejected."""
    lg = np.zeros((1, 8), np.float32)
    bad = [dict(k=1, G=3, S=1), dict(k=1, G=2, S=3), dict(k=9, G=1, S=1),
           dict(k=5, G=4, S=2), dict(k=1, G=8, S=1, two=True), dict(k=1, G=1, S=1, scale=0.0),
           dict(k=1, G=1, S=1, scale=math.inf), dict(k=65, G=1, S=1)]
    for a in bad:
        width = 128 if a["k"] == 65 else 8
        try:
            oracle.route_sigmoid_grouped(np.zeros((1, width), np.float32), "f32", None, a["k"],
                                         a["G"], a["S"], a.get("two", False), False,
                                         a.get("scale", 1.0), lib)
        except ValueError:
            continue
        raise AssertionError(f"accepted {a}")
    oracle.route_sigmoid_grouped(lg, "f32", None, 4, 4, 2, True, True, 1.0, lib)


def check_route_selection_sort(lib):
    """Brute force over heavy-tie rows: the selection equals a stable sort
    by (logit descending, id ascending) done by numpy."""
    rng = np.random.default_rng(12)
    for E in (2, 3, 5, 8, 31, 32, 33, 70):
        logits = rng.integers(-2, 3, size=(40, E)).astype(np.float32) * 0.5
        logits[::7, ::3] = -np.inf
        for k in sorted({1, 2, min(3, E), E // 2 or 1, E}):
            idx, _, _ = oracle.route(logits, "f32", k, False, lib)
            for t in range(logits.shape[0]):
                order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
                assert idx[t].tolist() == order[:k].tolist(), (E, k, t)


def check_route_weight_sums(lib):
    rng = np.random.default_rng(13)
    logits = rng.standard_normal((200, 64)).astype(np.float32)
    for k in (1, 2, 6, 64):
        _, w, _ = oracle.route(logits, "f32", k, True, lib)
        s = w.astype(np.float64).sum(axis=1)
        assert np.all(np.abs(s - 1.0) <= k * 2.0 ** -22 + 2 ** -23)
        _, w, _ = oracle.route(logits, "f32", k, False, lib)
        s = w.astype(np.float64).sum(axis=1)
        assert np.all(s <= 1.0 + 64 * 2.0 ** -23)
        assert np.all(w > 0)


def check_route_low_precision_logits(lib):
    """BF16/F16 logits: upcasting is exact, so routing them equals routing
    their FP32 values with the weights rounded once to the logits dtype."""
    rng = np.random.default_rng(14)
    base = rng.standard_normal((64, 16)).astype(np.float32)
    for dt in ("bf16", "f16"):
        low = oracle.convert(base, "f32", dt, lib)
        up = oracle.convert(low, dt, "f32", lib)
        for ren in (False, True):
            i1, w1, _ = oracle.route(low, dt, 4, ren, lib)
            i2, w2, _ = oracle.route(up, "f32", 4, ren, lib)
            assert np.array_equal(i1, i2)
            assert np.array_equal(w1, oracle.convert(w2, "f32", dt, lib))


def check_route_arguments(lib):
    x = np.zeros((2, 4), np.float32)
    for k in (0, 5):
        try:
            oracle.route(x, "f32", k, False, lib)
        except ValueError:
            continue
        raise AssertionError("top_k outside [1, E] must be rejected")


# ------------------------------------------------------------------- dispatch

def check_dispatch_invariants(lib):
    rng = np.random.default_rng(21)
    for (T, k, E) in ((1, 1, 1), (17, 2, 8), (100, 6, 64), (64, 8, 256)):
        idx = rng.integers(0, E, size=(T, k)).astype(np.uint32)
        counts, offsets, row_of, src_of, bad = oracle.dispatch(idx, E, lib)
        flat = idx.reshape(-1)
        assert bad == 0 and counts.sum() == T * k and offsets[0] == 0
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert np.array_equal(np.diff(offsets), counts)
        assert sorted(row_of.tolist()) == list(range(T * k))
        assert np.array_equal(src_of[row_of], np.arange(T * k))
        for e in range(E):
            seg = src_of[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)   # stable within the expert
    # bad indices get no row
    idx = np.array([[0, 9], [1, 1]], np.uint32)
    counts, offsets, row_of, src_of, bad = oracle.dispatch(idx, 2, lib)
    assert bad == 1 and row_of[1] == -1 and counts.tolist() == [1, 2]
    assert src_of[3] == -1


def check_gather(lib):
    rng = np.random.default_rng(22)
    T, k, E, H = 30, 3, 5, 24
    idx = rng.integers(0, E, size=(T, k)).astype(np.uint32)
    _, offsets, row_of, src_of, _ = oracle.dispatch(idx, E, lib)
    x = oracle.convert(rng.standard_normal((T, H)).astype(np.float32), "f32", "bf16", lib)
    xd = oracle.gather(x, "bf16", k, src_of, T * k, lib)
    for a in range(T * k):
        assert np.array_equal(xd[row_of[a]], x[a // k])


# -------------------------------------------------------------------- experts

def _dense_expert(x, wg, wu, wd):
    """Numpy matmul evaluation of one bias-free SwiGLU expert."""
    g = x @ wg.T
    u = x @ wu.T
    return (g * scipy.special.expit(g) * u) @ wd.T


def check_swiglu_golden(lib):
    for fields in _lines("swiglu_cases.txt"):
        H, I = (int(v) for v in fields[0].split())
        x = np.array([[float(v) for v in fields[1].split()]], np.float32)
        mats = []
        for f in fields[2:5]:
            mats.append(np.array([[float(v) for v in r.split()]
                                  for r in f.split(";")], np.float32)[None])
        gate, up, down = mats
        assert gate.shape == (1, I, H) and down.shape == (1, H, I)
        y = oracle.swiglu_rows(x, "f32", [0], gate, up, down, lib)
        want = [_eval(e) for e in fields[5].split()]
        np.testing.assert_allclose(y[0], want, rtol=1e-14, atol=1e-15)


def check_single_expert_dense(lib):
    """E = 1, top_k = 1: weight is exactly 1 and the chain reduces to the
    textbook dense SwiGLU FFN, evaluated here with numpy matmul."""
    rng = np.random.default_rng(31)
    T, H, I = 12, 40, 24
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, 1)).astype(np.float32)
    gate = (rng.standard_normal((1, I, H)) / math.sqrt(H)).astype(np.float32)
    up = (rng.standard_normal((1, I, H)) / math.sqrt(H)).astype(np.float32)
    down = (rng.standard_normal((1, H, I)) / math.sqrt(I)).astype(np.float32)
    for ren in (False, True):
        o = oracle.forward(x, "f32", lg, "f32", gate, up, down, 1, ren, lib)
        assert np.all(o["w"] == 1.0) and np.all(o["idx"] == 0)
        ref = _dense_expert(x.astype(np.float64), gate[0].astype(np.float64),
                            up[0].astype(np.float64), down[0].astype(np.float64))
        np.testing.assert_allclose(o["y"], ref, rtol=1e-12, atol=1e-13)


def check_dense_brute_force(lib):
    """Evaluate every expert on every token densely (numpy), mask by the
    routing, and compare with the dispatched chain, for all top_k."""
    rng = np.random.default_rng(32)
    for (T, H, I, E) in ((16, 8, 6, 8), (9, 16, 12, 3), (5, 4, 4, 1)):
        x = rng.standard_normal((T, H)).astype(np.float32)
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[0, :] = np.nan if T > 3 else lg[0, :]
        gate = rng.standard_normal((E, I, H)).astype(np.float32) / 3
        up = rng.standard_normal((E, I, H)).astype(np.float32) / 3
        down = rng.standard_normal((E, H, I)).astype(np.float32) / 3
        dense = np.stack([_dense_expert(x.astype(np.float64),
                                        gate[e].astype(np.float64),
                                        up[e].astype(np.float64),
                                        down[e].astype(np.float64))
                          for e in range(E)])      # [E, T, H]
        for k in range(1, E + 1):
            for ren in (False, True):
                o = oracle.forward(x, "f32", lg, "f32", gate, up, down, k, ren, lib)
                mask = np.zeros((T, E))
                for t in range(T):
                    for j in range(k):
                        mask[t, o["idx"][t, j]] += float(o["w"][t, j])
                ref = np.einsum("te,eth->th", mask, dense)
                np.testing.assert_allclose(o["y"], ref, rtol=1e-11, atol=1e-12)


def check_linearity_and_permutation(lib):
    rng = np.random.default_rng(33)
    T, H, I, E, k = 20, 16, 8, 4, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    gate = rng.standard_normal((E, I, H)).astype(np.float32) / 4
    up = rng.standard_normal((E, I, H)).astype(np.float32) / 4
    down = rng.standard_normal((E, H, I)).astype(np.float32) / 4
    base = oracle.forward(x, "f32", lg, "f32", gate, up, down, k, True, lib)["y"]
    doubled = oracle.forward(x, "f32", lg, "f32", gate, up, down * 2, k, True, lib)["y"]
    assert np.array_equal(doubled, 2 * base), "scaling Wd by 2 must double y"
    perm = rng.permutation(T)
    py = oracle.forward(x[perm], "f32", lg[perm], "f32", gate, up, down, k, True, lib)["y"]
    assert np.array_equal(py, base[perm]), "permuting tokens must permute y"
    sub = oracle.forward_tokens([3, 11, 19], x, "f32", lg, "f32", gate, up, down,
                                k, True, lib)[2]
    np.testing.assert_allclose(sub, base[[3, 11, 19]], rtol=1e-13, atol=1e-14)


def check_exact_integer(lib):
    """Small integers keep every product and sum exact in double, and the
    gate values are chosen where SiLU is exact (g = 0 gives h = 0)."""
    T, H, I, E = 4, 3, 2, 2
    x = np.array([[1, 2, 0], [0, 1, 1], [2, 0, -1], [1, 1, 1]], np.float32)
    lg = np.array([[0, 1], [1, 0], [0, 2], [3, 0]], np.float32)
    gate = np.zeros((E, I, H), np.float32)       # g = 0 -> SiLU(g) = 0
    up = np.ones((E, I, H), np.float32)
    down = np.ones((E, H, I), np.float32)
    o = oracle.forward(x, "f32", lg, "f32", gate, up, down, 1, True, lib)
    assert np.array_equal(o["y"], np.zeros((T, H)))
    assert o["idx"].reshape(-1).tolist() == [1, 0, 1, 0]


# -------------------------------------------------------------------- combine

def check_combine_one_hot(lib):
    """With weights one-hot per token the combine is an exact gather of the
    selected expert row; zero weights remove a row entirely."""
    rng = np.random.default_rng(41)
    T, k, H = 10, 3, 12
    out = rng.standard_normal((T * k, H)).astype(np.float32)
    row_of = rng.permutation(T * k).astype(np.int32)
    w = np.zeros((T, k), np.float32)
    pick = rng.integers(0, k, size=T)
    w[np.arange(T), pick] = 1.0
    y = oracle.combine(out, "f32", w, "f32", row_of, k, lib)
    for t in range(T):
        assert np.array_equal(y[t], out[row_of[t * k + pick[t]]].astype(np.float64))
    row_of[4] = -1
    y = oracle.combine(out, "f32", w, "f32", row_of, k, lib)
    assert np.isnan(y[1]).all() and not np.isnan(y[0]).any()


def check_combine_weighted(lib):
    T, k, H = 3, 2, 2
    out = np.array([[1, 2], [3, 4], [5, 6], [7, 8], [9, 10], [11, 12]], np.float32)
    row_of = np.array([5, 0, 1, 2, 3, 4], np.int32)
    w = np.array([[0.5, 0.25], [1, -1], [2, 0]], np.float32)
    y = oracle.combine(out, "f32", w, "f32", row_of, k, lib)
    assert y.tolist() == [[0.5 * 11 + 0.25 * 1, 0.5 * 12 + 0.25 * 2],
                          [3 - 5, 4 - 6], [2 * 7, 2 * 8]]


# -------------------------------------------------------------------- rmsnorm

def check_combine_v2_hand_cases(lib):
    """aclnnMoeDistributeCombineAddRmsNormV2 (formula and parameter list):
    special experts by id range after the E routed experts, the shared-expert
    term inside the sum over slots, and the active mask. Each case is worked
    by hand (H = 2)."""
    f = np.float32
    cv = lambda out, w, rows, k, **kw: oracle.combine_v2(
        np.array(out, f), "f32", np.array(w, f), "f32", np.array(rows, np.int32), k, "f32",
        lib=lib, **{n: (np.array(v, f) if n in ("ori_x", "alpha1", "alpha2", "const_v",
                                                  "shared_x") else v) for n, v in kw.items()})
    out = [[1, 2], [0, 1]]
    # zero expert (id 2 with E=2, zero=1): 0.5*[1,2] + 0.5*0
    y = cv(out, [[0.5, 0.5]], [0, -1], 2, ids=[[0, 2]], E=2, zero=1)
    assert y.tolist() == [[0.5, 1.0]]
    # copy expert (E=2, zero=1, copy=1 -> id 3): 0.25 * oriX
    y = cv(out, [[0.25]], [-1], 1, ids=[[3]], E=2, zero=1, copy=1, ori_x=[[4, -2]])
    assert y.tolist() == [[1.0, -0.5]]
    # const expert c = 1 (E=2, const=2 -> ids 2, 3): 0.5*(2*[1,2] + 3*[1,1])
    y = cv(out, [[0.5]], [-1], 1, ids=[[3]], E=2, const=2, ori_x=[[1, 2]], alpha1=[7, 2],
           alpha2=[5, 3], const_v=[[9, 9], [1, 1]])
    assert y.tolist() == [[2.5, 3.5]]
    # shared expert, weights summing to 1/2: [0.25,0.25] + (0.25+0.25)*[8,4]
    y = cv([[1, 0], [0, 1]], [[0.25, 0.25]], [0, 1], 2, shared_x=[[8, 4]])
    assert y.tolist() == [[4.25, 2.25]]
    # 2-D mask keeps slot 0 only, shared term included for it: 0.25*[1,0] + 0.25*[8,4]
    y = cv([[1, 0], [0, 1]], [[0.25, 0.75]], [0, 1], 2, shared_x=[[8, 4]],
           mask=np.array([[True, False]]))
    assert y.tolist() == [[2.25, 1.0]]
    # 1-D mask drops token 1 entirely (no shared term either)
    y = cv([[1, 0], [0, 1]], [[1.0], [1.0]], [0, 1], 1, shared_x=[[8, 4], [8, 4]],
           mask=np.array([True, False]))
    assert y.tolist() == [[9.0, 4.0], [0.0, 0.0]]
    # an id past the last special expert, or a routed id without a row: NaN
    y = cv(out, [[1.0]], [0], 1, ids=[[5]], E=2, zero=1, copy=1, ori_x=[[3, 3]])
    assert np.isnan(y).all()
    y = cv(out, [[1.0]], [-1], 1, ids=[[1]], E=2, zero=1)
    assert np.isnan(y).all()
    # a 1-D mask that keeps a token after a dropped one is rejected
    try:
        cv(out, [[1.0], [1.0]], [0, 1], 1, mask=np.array([False, True]))
    except ValueError:
        pass
    else:
        raise AssertionError("1-D mask order not enforced")


def check_combine_v2_invariants(lib):
    """Random inputs: with no extras it is the (separately pinned) combine;
    a const expert with alpha = (1, 0) is a copy expert; a masked slot is a
    slot of weight 0; with weights renormalised to 1 the shared expert adds
    its row once."""
    rng = np.random.default_rng(17)
    T, k, H, E = 9, 3, 12, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w, _ = oracle.route(logits, "f32", k, True, lib)
    _, _, row_of, _, _ = oracle.dispatch(idx, E, lib)
    out = rng.standard_normal((T * k, H)).astype(np.float32)
    base = oracle.combine(out, "f32", w, "f32", row_of, k, lib)
    y = oracle.combine_v2(out, "f32", w, "f32", row_of, k, "f32", lib=lib)
    assert np.array_equal(y, base)
    shared = rng.standard_normal((T, H)).astype(np.float32)
    y = oracle.combine_v2(out, "f32", w, "f32", row_of, k, "f32", shared_x=shared, lib=lib)
    assert np.allclose(y, base + shared.astype(np.float64), rtol=1e-6, atol=1e-6)
    mask = rng.random((T, k)) < 0.6
    y = oracle.combine_v2(out, "f32", w, "f32", row_of, k, "f32", mask=mask, lib=lib)
    w0 = np.where(mask, w, np.float32(0))
    assert np.allclose(y, oracle.combine(out, "f32", w0, "f32", row_of, k, lib), rtol=1e-12,
                       atol=1e-12)
    ori = rng.standard_normal((T, H)).astype(np.float32)
    ids = idx.copy()
    ids[:, 1] = E + 1                      # copy expert (zero=1, copy=1) vs const with (1, 0)
    a = oracle.combine_v2(out, "f32", w, "f32", row_of, k, "f32", ids=ids, E=E, zero=1,
                          copy=1, ori_x=ori, lib=lib)
    ids[:, 1] = E + 1                      # const expert 0 (zero=1, copy=0)
    b = oracle.combine_v2(out, "f32", w, "f32", row_of, k, "f32", ids=ids, E=E, zero=1,
                          const=1, ori_x=ori, alpha1=np.ones(1, np.float32),
                          alpha2=np.zeros(1, np.float32), const_v=np.full((1, H), 7, np.float32),
                          lib=lib)
    assert np.array_equal(a, b)


def check_rmsnorm_golden(lib):
    for fields in _lines("rmsnorm_cases.txt"):
        H = int(fields[0].split()[0])
        eps = float(fields[0].split()[1])
        comb = np.array([[float(v) for v in fields[1].split()]], np.float64)
        res = np.array([[float(v) for v in fields[2].split()]], np.float32)
        gamma = np.array([float(v) for v in fields[3].split()], np.float32)
        y, xo, rstd = oracle.add_rmsnorm(comb, res, "f32", gamma, "f32", eps, lib)
        assert xo[0].tolist() == [float(v) for v in fields[4].split()]
        r = _eval(fields[5], eps=eps)
        assert _f32_close(float(rstd[0]), r, 1e-7)
        want = [_eval(e, eps=eps, rstd=r) for e in fields[6].split()]
        np.testing.assert_allclose(y[0].astype(np.float64), want, rtol=2e-7, atol=1e-30)
        assert xo.shape == (1, H)


def check_rmsnorm_constant_rows(lib):
    """Constant row c: y = sign(c) * gamma / sqrt(1 + eps / c^2)."""
    rng = np.random.default_rng(51)
    H = 96
    gamma = (1 + 0.3 * rng.standard_normal(H)).astype(np.float32)
    cs = np.array([-3.0, -0.25, 0.5, 1.0, 7.0], np.float32)
    x = np.repeat(cs[:, None], H, axis=1)
    for eps in (1e-6, 1e-2, 1.0):
        y, rstd = oracle.rmsnorm(x, "f32", gamma, "f32", eps, lib=lib)
        for i, c in enumerate(cs.astype(np.float64)):
            want = np.sign(c) * gamma / math.sqrt(1 + eps / c ** 2)
            np.testing.assert_allclose(y[i], want, rtol=3e-7)
            assert _f32_close(float(rstd[i]), 1 / math.sqrt(c * c + eps), 1e-7)


def check_add_rmsnorm_is_rmsnorm_of_xout(lib):
    rng = np.random.default_rng(52)
    T, H = 7, 64
    comb = rng.standard_normal((T, H))
    res = oracle.convert(rng.standard_normal((T, H)).astype(np.float32), "f32", "bf16", lib)
    gamma = oracle.convert((1 + 0.3 * rng.standard_normal(H)).astype(np.float32), "f32", "bf16", lib)
    y, xo, rstd = oracle.add_rmsnorm(comb, res, "bf16", gamma, "bf16", 1e-6, lib)
    xr = oracle.to_f64(res, "bf16", lib) + comb
    assert np.array_equal(xo, oracle.convert(xr, "f64", "bf16", lib))
    y2, rstd2 = oracle.rmsnorm(xo, "bf16", gamma, "bf16", 1e-6, lib=lib)
    assert np.array_equal(y, y2) and np.array_equal(rstd, rstd2)
    # numpy statement of the normalisation on the rounded x
    xf = oracle.to_f64(xo, "bf16", lib)
    r = 1 / np.sqrt((xf ** 2).mean(axis=1) + 1e-6)
    np.testing.assert_allclose(rstd, r, rtol=1e-7)


def check_rmsnorm_eps_validation(lib):
    x = np.ones((1, 4), np.float32)
    g = np.ones(4, np.float32)
    for eps in (0.0, -1.0, math.inf, math.nan):
        try:
            oracle.rmsnorm(x, "f32", g, "f32", eps, lib=lib)
        except ValueError:
            continue
        raise AssertionError(f"eps={eps} must be rejected")


from oracle_pins_training import *  # noqa: E402,F401,F403  (the training pins)

ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
