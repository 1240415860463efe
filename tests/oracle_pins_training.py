"""Pins of the first-order training part of the CPU oracle (ruDNN user guide,
section 12 "MoE first-order training") to facts fixed outside the oracle.

Each ``check_*`` takes a loaded oracle library and raises ``AssertionError``
when the oracle disagrees with:

* library routines the weights reduce to (``scipy.special.softmax`` and
  ``scipy.special.expit`` on the selected logits);
* central finite differences of the oracle's own forward functions, each of
  which is pinned separately (router weights here; the SwiGLU experts and the
  combine in ``oracle_pins.py``) -- the derivative is a fact of the forward,
  not of the backward's code;
* torch autograd (float64, CPU) of a dense SwiGLU written with torch ops;
* exact invariants: the adjoint identity of the dispatch gather on integer
  data, shift invariance of the softmax, zero gradient outside the selection
  for the sigmoid and for the renormalised softmax, linearity in the scale.
"""

from __future__ import annotations

import numpy as np
import scipy.special
import torch

import oracle


def _rel_close(a, b, rel, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    err = np.max(np.abs(a - b)) / scale
    assert err <= rel, f"{what}: relative error {err:.3e} > {rel:.1e}"


def _rows_nan(a):
    return np.isnan(np.asarray(a, dtype=np.float64)).all(axis=1)


# ---- router weights --------------------------------------------------------

def check_router_weights_library(lib):
    rng = np.random.default_rng(11)
    T, E = 6, 9
    logits = rng.standard_normal((T, E)) * 2.0
    idx = np.stack([rng.permutation(E)[:4] for _ in range(T)])
    l32 = logits.astype(np.float32)
    # softmax over all experts, every expert selected in id order: the library softmax
    w, n = oracle.router_weights(l32, "f32", np.tile(np.arange(E), (T, 1)), "softmax",
                                 False, 1.0, "f64", lib)
    assert n == 0
    _rel_close(w, scipy.special.softmax(l32.astype(np.float64), axis=1), 1e-12, "softmax k=E")
    for scale in (1.0, 2.5):
        # renormalised softmax of a selection = softmax of the selected logits alone
        w, _ = oracle.router_weights(l32, "f32", idx, "softmax", True, scale, "f64", lib)
        sel = np.take_along_axis(l32.astype(np.float64), idx, axis=1)
        _rel_close(w, scale * scipy.special.softmax(sel, axis=1), 1e-12, "renorm softmax")
        # plain softmax of a selection: the selected entries of the full softmax
        w, _ = oracle.router_weights(l32, "f32", idx, "softmax", False, scale, "f64", lib)
        full = scipy.special.softmax(l32.astype(np.float64), axis=1)
        _rel_close(w, scale * np.take_along_axis(full, idx, axis=1), 1e-12, "softmax")
        # sigmoid scores, plain and renormalised
        w, _ = oracle.router_weights(l32, "f32", idx, "sigmoid", False, scale, "f64", lib)
        _rel_close(w, scale * scipy.special.expit(sel), 1e-12, "sigmoid")
        w, _ = oracle.router_weights(l32, "f32", idx, "sigmoid", True, scale, "f64", lib)
        s = scipy.special.expit(sel)
        _rel_close(w, scale * s / s.sum(axis=1, keepdims=True), 1e-12, "renorm sigmoid")
    # FP32 output is the f64 result rounded once
    w64, _ = oracle.router_weights(l32, "f32", idx, "softmax", True, 1.0, "f64", lib)
    w32, _ = oracle.router_weights(l32, "f32", idx, "softmax", True, 1.0, "f32", lib)
    assert np.array_equal(w32, w64.astype(np.float32))


def check_router_weights_gather_and_nan_rules(lib):
    logits = np.array([[0.5, -1.0, 2.0, 0.0],
                       [0.5, -1.0, 2.0, 0.0],
                       [0.5, -1.0, 2.0, 0.0],
                       [0.5, -1.0, 2.0, 0.0],
                       [np.nan, 0.0, 1.0, 2.0],
                       [np.inf, 0.0, 1.0, 2.0],
                       [-np.inf] * 4,
                       [-np.inf, 0.0, 1.0, 2.0]], dtype=np.float32)
    idx = np.array([[2, 2, 0], [0, 1, 4], [0, 1, 2], [3, -1, 0], [1, 2, 3], [1, 2, 3],
                    [0, 1, 2], [0, 1, 2]], dtype=np.int64)
    p = scipy.special.softmax(logits[0].astype(np.float64))
    w, n = oracle.router_weights(logits, "f32", idx, "softmax", False, 1.0, "f64", lib)
    # a repeated id is gathered again (row 0)
    assert np.allclose(w[0], [p[2], p[2], p[0]], rtol=1e-14, atol=0)
    # ids outside [0, E) make the row NaN (rows 1, 3); others untouched (row 2)
    assert _rows_nan(w).tolist() == [False, True, False, True, True, True, True, False]
    assert n == 5
    # a -inf logit is a valid row with score 0 (row 7)
    assert w[7, 0] == 0.0 and np.all(np.isfinite(w[7]))
    # renormalised duplicates: each copy counts in the sum
    w, _ = oracle.router_weights(logits[:1], "f32", idx[:1], "softmax", True, 1.0, "f64", lib)
    z = 2 * p[2] + p[0]
    assert np.allclose(w[0], [p[2] / z, p[2] / z, p[0] / z], rtol=1e-14, atol=0)
    # sigmoid: +-inf logits are valid scores 1 and 0; a NaN only where selected
    lg = np.array([[np.inf, -np.inf, np.nan, 0.0]], dtype=np.float32)
    w, n = oracle.router_weights(lg, "f32", np.array([[0, 1, 3]]), "sigmoid", False, 2.0,
                                 "f64", lib)
    assert n == 0 and w.tolist() == [[2.0, 0.0, 1.0]]
    # unsigned ids: 2^32 - 1 is illegal, never wrapped to a valid id
    w, n = oracle.router_weights(logits[:1], "f32",
                                 np.array([[0, 1, 0xFFFFFFFF]], dtype=np.uint32), "softmax",
                                 False, 1.0, "f64", lib)
    assert n == 1 and _rows_nan(w)[0]
    # argument limits of the section
    for kw in (dict(scale=0.0), dict(scale=-1.0), dict(scale=np.inf), dict(scale=np.nan)):
        try:
            oracle.router_weights(logits[:1], "f32", idx[2:3], "softmax", False,
                                  kw["scale"], "f64", lib)
        except ValueError:
            continue
        raise AssertionError(f"scale {kw['scale']} accepted")
    try:
        oracle.router_weights(np.zeros((1, 70), np.float32), "f32",
                              np.arange(65)[None, :], "softmax", False, 1.0, "f64", lib)
    except ValueError:
        pass
    else:
        raise AssertionError("top_k = 65 accepted")


# ---- router backward -------------------------------------------------------

def _fd_router(lib, logits, idx, gw, scoring, renorm, scale, h=1e-6):
    T, E = logits.shape
    g = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            lp = logits.copy(); lp[t, e] += h
            lm = logits.copy(); lm[t, e] -= h
            wp, _ = oracle.router_weights(lp, "f64", idx, scoring, renorm, scale, "f64", lib)
            wm, _ = oracle.router_weights(lm, "f64", idx, scoring, renorm, scale, "f64", lib)
            g[t, e] = np.sum(gw[t] * (wp[t] - wm[t])) / (2 * h)
    return g


def check_router_backward_finite_differences(lib):
    rng = np.random.default_rng(12)
    T, E, k = 4, 7, 3
    logits = rng.standard_normal((T, E)) * 1.5
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    idx[1] = [4, 4, 2]  # a repeated id
    gw = rng.standard_normal((T, k))
    for scoring in ("softmax", "sigmoid"):
        for renorm in (False, True):
            for scale in (1.0, 2.5):
                dl, n = oracle.router_backward(logits, "f64", idx, gw, "f64", scoring, renorm,
                                               scale, "f64", lib)
                assert n == 0
                fd = _fd_router(lib, logits, idx, gw, scoring, renorm, scale)
                _rel_close(dl, fd, 1e-7, f"router backward {scoring} renorm={renorm} "
                                         f"scale={scale}")


def check_router_backward_invariants(lib):
    rng = np.random.default_rng(13)
    T, E, k = 8, 10, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    gw = rng.standard_normal((T, k)).astype(np.float32)
    unsel = np.ones((T, E), bool)
    np.put_along_axis(unsel, idx, False, axis=1)
    # softmax without renormalisation: adding a constant to a row changes nothing
    dl, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "softmax", False, 1.0,
                                   "f64", lib)
    assert np.all(np.abs(dl.sum(axis=1)) <= 1e-12 * np.abs(dl).sum(axis=1))
    assert np.all(np.abs(dl[unsel]) > 0)
    # renormalised softmax depends on the selected logits only
    dl, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "softmax", True, 1.0,
                                   "f64", lib)
    assert np.max(np.abs(dl[unsel])) <= 1e-14 * np.max(np.abs(dl))
    assert np.all(np.abs(dl.sum(axis=1)) <= 1e-12 * np.abs(dl).sum(axis=1))
    # sigmoid: exactly zero outside the selection
    for renorm in (False, True):
        dl, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "sigmoid", renorm, 1.0,
                                       "f64", lib)
        assert np.all(dl[unsel] == 0.0) and np.all(dl[~unsel] != 0.0)
    # a NaN logit outside a sigmoid selection leaves the gradient untouched
    lg = logits.copy(); lg[0, unsel[0].nonzero()[0][0]] = np.nan
    d_nan, n = oracle.router_backward(lg, "f32", idx, gw, "f32", "sigmoid", True, 1.0, "f64",
                                      lib)
    d_ref, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "sigmoid", True, 1.0,
                                      "f64", lib)
    assert n == 0 and np.array_equal(d_nan, d_ref)
    # linear in the scale, with and without renormalisation
    for scoring in ("softmax", "sigmoid"):
        for renorm in (False, True):
            a, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", scoring, renorm, 1.0,
                                          "f64", lib)
            b, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", scoring, renorm, 3.0,
                                          "f64", lib)
            _rel_close(b, 3.0 * a, 1e-14, "scale linearity")
    # output dtype: the f64 gradient rounded once (bf16 via float32, as torch does)
    d64, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "softmax", True, 1.0,
                                    "f64", lib)
    d32, _ = oracle.router_backward(logits, "f32", idx, gw, "f32", "softmax", True, 1.0,
                                    "f32", lib)
    assert np.array_equal(d32, d64.astype(np.float32))
    lb = torch.from_numpy(logits).to(torch.bfloat16)
    lbits = lb.view(torch.int16).numpy().view(np.uint16)
    db, _ = oracle.router_backward(lbits, "bf16", idx, gw, "f32", "softmax", False, 1.0,
                                   None, lib)
    d64b, _ = oracle.router_backward(lbits, "bf16", idx, gw, "f32", "softmax", False, 1.0,
                                     "f64", lib)
    ref = torch.from_numpy(d64b.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(db, ref.view(torch.int16).numpy().view(np.uint16))
    # an illegal id NaNs the row and only that row
    bad = idx.copy(); bad[3, 1] = E
    dl, n = oracle.router_backward(logits, "f32", bad, gw, "f32", "softmax", False, 1.0,
                                   "f64", lib)
    assert n == 1 and _rows_nan(dl).tolist() == [t == 3 for t in range(T)]


# ---- combine backward ------------------------------------------------------

def check_combine_backward_exact(lib):
    """The combine is bilinear in (expert outputs, weights): on small integers
    a unit step of one input changes <gy, y> by exactly that input's
    gradient."""
    rng = np.random.default_rng(14)
    T, k, H = 5, 3, 4
    rows = T * k
    row_of = rng.permutation(rows).astype(np.int32)
    out = rng.integers(-4, 5, (rows, H)).astype(np.float64)
    w = rng.integers(-3, 4, (T, k)).astype(np.float64)
    gy = rng.integers(-3, 4, (T, H)).astype(np.float64)
    dexp, dw = oracle.combine_backward(out, "f64", w, "f64", row_of, gy, "f64", k, lib)

    def loss(o, ww):
        return float(np.sum(gy * oracle.combine(o, "f64", ww, "f64", row_of, k, lib)))

    base = loss(out, w)
    for r in range(rows):
        for h in range(H):
            o2 = out.copy(); o2[r, h] += 1.0
            assert loss(o2, w) - base == dexp[r, h], ("dexpert", r, h)
    for t in range(T):
        for j in range(k):
            w2 = w.copy(); w2[t, j] += 1.0
            assert loss(out, w2) - base == dw[t, j], ("dw", t, j)
    # a slot with no row: its dw is NaN, the token's other slots are unaffected
    ro = row_of.copy(); dropped = ro[4]; ro[4] = -1
    dexp2, dw2 = oracle.combine_backward(out, "f64", w, "f64", ro, gy, "f64", k, lib)
    assert np.isnan(dw2[1, 1]) and np.array_equal(np.delete(dw2.ravel(), 4),
                                                  np.delete(dw.ravel(), 4))
    assert np.all(dexp2[dropped] == 0.0)


# ---- SwiGLU expert backward ------------------------------------------------

def check_swiglu_backward_finite_differences(lib):
    rng = np.random.default_rng(15)
    E, H, I, n = 2, 3, 2, 4
    x = rng.standard_normal((n, H))
    gate = rng.standard_normal((E, I, H))
    up = rng.standard_normal((E, I, H))
    down = rng.standard_normal((E, H, I))
    eor = np.array([1, 0, 1, 1], dtype=np.int32)
    dout = rng.standard_normal((n, H))
    dx, dg, du, dd = oracle.swiglu_backward_rows(x, "f64", eor, gate, up, down, dout, "f64",
                                                 lib)
    h = 1e-6

    def loss(xx, gg, uu, ddn):
        return float(np.sum(dout * oracle.swiglu_rows(xx, "f64", eor, gg, uu, ddn, lib)))

    args = [x, gate, up, down]
    for which, grad in enumerate((dx, dg, du, dd)):
        fd = np.zeros_like(grad)
        for pos in np.ndindex(*grad.shape):
            ap = [a.copy() for a in args]; am = [a.copy() for a in args]
            ap[which][pos] += h; am[which][pos] -= h
            fd[pos] = (loss(*ap) - loss(*am)) / (2 * h)
        _rel_close(grad, fd, 1e-7, f"swiglu backward operand {which}")


def check_swiglu_backward_autograd(lib):
    """Against torch autograd of a dense SwiGLU written with torch ops."""
    rng = np.random.default_rng(16)
    E, H, I, n = 3, 16, 8, 9
    x = rng.standard_normal((n, H))
    gate = rng.standard_normal((E, I, H)) / 4
    up = rng.standard_normal((E, I, H)) / 4
    down = rng.standard_normal((E, H, I)) / 3
    eor = rng.integers(0, E, n).astype(np.int32)
    dout = rng.standard_normal((n, H))
    dx, dg, du, dd = oracle.swiglu_backward_rows(x, "f64", eor, gate, up, down, dout, "f64",
                                                 lib)
    tx = torch.tensor(x, requires_grad=True)
    tg = torch.tensor(gate, requires_grad=True)
    tu = torch.tensor(up, requires_grad=True)
    td = torch.tensor(down, requires_grad=True)
    te = torch.tensor(eor, dtype=torch.long)
    a = torch.einsum("nih,nh->ni", tg[te], tx)
    b = torch.einsum("nih,nh->ni", tu[te], tx)
    o = torch.einsum("nhi,ni->nh", td[te], torch.nn.functional.silu(a) * b)
    (o * torch.tensor(dout)).sum().backward()
    for got, ref, name in ((dx, tx.grad, "dx"), (dg, tg.grad, "dgate"), (du, tu.grad, "dup"),
                           (dd, td.grad, "ddown")):
        _rel_close(got, ref.numpy(), 1e-12, f"autograd {name}")


# ---- dispatch backward -----------------------------------------------------

def check_dispatch_backward_adjoint(lib):
    """The gather x -> x_disp is linear; its backward is its adjoint:
    <gather(x), d> = <x, dispatch_backward(d)>, exact on integers."""
    rng = np.random.default_rng(17)
    T, E, k, H = 9, 5, 3, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.uint32)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E, lib)
    x = rng.integers(-5, 6, (T, H)).astype(np.float32)
    xd = oracle.gather(x, "f32", k, src_of, T * k, lib)
    d = rng.integers(-5, 6, (T * k, H)).astype(np.float32)
    dx = oracle.dispatch_backward(d, "f32", row_of, k, lib)
    assert float(np.sum(xd.astype(np.float64) * d)) == float(np.sum(x.astype(np.float64) * dx))
    # unit test vectors: every token gets exactly its k rows, unweighted
    for t in range(T):
        assert np.array_equal(dx[t], d[row_of[t * k:(t + 1) * k]].astype(np.float64).sum(0))
    # a slot with no row adds nothing
    ro = row_of.copy(); r = ro[5]; ro[5] = -1
    dx2 = oracle.dispatch_backward(d, "f32", ro, k, lib)
    assert np.array_equal(dx2[1], dx[1] - d[r])


# ---- the whole backward chain ----------------------------------------------

def check_training_chain_finite_differences(lib):
    """<gy, y> of the full forward (fixed selection, router weights, dispatch,
    experts, combine) differentiated numerically, against the four backward
    steps chained in the section's order."""
    rng = np.random.default_rng(18)
    T, E, k, H, I = 5, 4, 2, 3, 2
    logits = rng.standard_normal((T, E))
    x = rng.standard_normal((T, H))
    gate = rng.standard_normal((E, I, H))
    up = rng.standard_normal((E, I, H))
    down = rng.standard_normal((E, H, I))
    gy = rng.standard_normal((T, H))
    idx, _, _ = oracle.route(logits.astype(np.float32), "f32", k, False, lib)
    counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E, lib)

    def forward(lg, xx, gg, uu, dd):
        w, _ = oracle.router_weights(lg, "f64", idx, "softmax", True, 1.5, "f64", lib)
        xd = oracle.gather(xx, "f64", k, src_of, T * k, lib)
        out = oracle.experts_dispatched(xd, "f64", offsets, gg, uu, dd, lib)
        return w, xd, out, oracle.combine(out, "f64", w, "f64", row_of, k, lib)

    w, xd, out, y = forward(logits, x, gate, up, down)
    dexp, dw = oracle.combine_backward(out, "f64", w, "f64", row_of, gy, "f64", k, lib)
    dxd, dg, du, dd = oracle.experts_backward_dispatched(xd, "f64", offsets, gate, up, down,
                                                         dexp, "f64", lib)
    dx = oracle.dispatch_backward(dxd, "f64", row_of, k, lib)
    dl, _ = oracle.router_backward(logits, "f64", idx, dw, "f64", "softmax", True, 1.5,
                                   "f64", lib)
    args = [logits, x, gate, up, down]
    h = 1e-6
    for which, grad in enumerate((dl, dx, dg, du, dd)):
        fd = np.zeros_like(grad)
        for pos in np.ndindex(*grad.shape):
            ap = [a.copy() for a in args]; am = [a.copy() for a in args]
            ap[which][pos] += h; am[which][pos] -= h
            fd[pos] = (np.sum(gy * forward(*ap)[3]) - np.sum(gy * forward(*am)[3])) / (2 * h)
        _rel_close(grad, fd, 2e-7, f"chain operand {which}")


def check_swiglu_cache_matches_forward(lib):
    """The cache's h equals the forward's SwiGLU activation: pushed through a
    down projection of ones it must give the forward's output."""
    rng = np.random.default_rng(19)
    E, H, I, n = 3, 8, 5, 7
    x = rng.standard_normal((n, H))
    gate = rng.standard_normal((E, I, H))
    up = rng.standard_normal((E, I, H))
    counts = np.array([2, 0, 5])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    g, u, h = oracle.experts_cache_dispatched(x, "f64", offsets, gate, up, lib)
    owner = np.repeat(np.arange(E), counts)
    # g and u are the plain products (numpy matmul per row)
    for r in range(n):
        assert np.allclose(g[r], gate[owner[r]] @ x[r], rtol=1e-13, atol=1e-13)
        assert np.allclose(u[r], up[owner[r]] @ x[r], rtol=1e-13, atol=1e-13)
    # h against the forward: a down projection with unit vectors reads h back
    for i in range(I):
        down = np.zeros((E, H, I)); down[:, 0, i] = 1.0
        out = oracle.experts_dispatched(x, "f64", offsets.astype(np.int32), gate, up, down, lib)
        assert np.allclose(out[:, 0], h[:, i], rtol=1e-14, atol=0)


def check_swiglu_backward_column_restriction(lib):
    """The full-size training test reads an expert's weight gradients at a few
    intermediate columns from the backward of the expert restricted to those
    columns (rows of Wg / Wu, columns of Wd). In a SwiGLU FFN column i
    touches only row i of Wg / Wu and column i of Wd, so the restricted
    backward's weight gradients equal the full one's at those columns, bit for
    bit, for any input dtype."""
    rng = np.random.default_rng(23)
    H, I, n = 24, 20, 11
    cols = [0, 7, 19]
    for dt in ("f64", "bf16"):
        x = rng.standard_normal((n, H))
        gate = rng.standard_normal((1, I, H)) / 4
        up = rng.standard_normal((1, I, H)) / 4
        down = rng.standard_normal((1, H, I)) / 3
        dout = rng.standard_normal((n, H))
        if dt == "bf16":
            x, gate, up, down = (oracle.convert(a.astype(np.float32), "f32", "bf16", lib)
                                 for a in (x, gate, up, down))
        eor = np.zeros(n, np.int32)
        _, dg, du, dd = oracle.swiglu_backward_rows(x, dt, eor, gate, up, down, dout, "f64", lib)
        gs = np.ascontiguousarray(gate[:, cols, :])
        us = np.ascontiguousarray(up[:, cols, :])
        ds = np.ascontiguousarray(down[:, :, cols])
        _, dgs, dus, dds = oracle.swiglu_backward_rows(x, dt, eor, gs, us, ds, dout, "f64", lib)
        assert np.array_equal(dgs[0], dg[0][cols, :]), f"{dt}: gate gradient rows"
        assert np.array_equal(dus[0], du[0][cols, :]), f"{dt}: up gradient rows"
        assert np.array_equal(dds[0], dd[0][:, cols]), f"{dt}: down gradient columns"
