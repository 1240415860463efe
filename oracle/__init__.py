"""Plain CPU oracle for the local Mixture-of-Experts FFN forward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``mixture_experts_ffn_topk_gb300``) never imports
it, and this package imports nothing from the product path.

The arithmetic lives in ``moe_oracle.c`` (plain C loops, FP32 routing as the
ruDNN routing contract fixes it, double everywhere else); this module compiles
it with gcc on first use and marshals numpy arrays through ctypes.

Arrays: f32 data is ``np.float32``; bf16 and f16 data are raw 16-bit words in
``np.uint16`` arrays (``np.float16`` is accepted for f16); f64 is
``np.float64``. Functions return numpy arrays in the same conventions.

Sources, by page title and section:
  ruDNN user guide, sections 3-7 (MoE workflow, routing contract, expert
  weights and dispatch, calling MoE, RMSNorm), section 10 (grouped sigmoid
  routing) and section 12 (MoE first-order training); aclnnMoeDistributeCombine-
  AddRmsNormV2, "Function" formula (combine, Add, RMSNorm, rstdOut);
  aclnnFFN, "Formula" (the FFN the experts instantiate).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2, "f64": 3}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_F = ctypes.c_float


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``oracle/_build/liboracle.so``.

    Plain ``-O2``: no fast-math (which would change NaN handling and rounding),
    no vector intrinsics, portable across x86_64 and aarch64.
    """
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` overrides it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    lib.oracle_convert.argtypes = [_P, _INT, _P, _INT, _I64]
    lib.oracle_convert.restype = None
    lib.oracle_route.argtypes = [_P, _INT, _I64, _I64, _I64, _INT, _P, _P]
    lib.oracle_route.restype = _I64
    lib.oracle_route_sigmoid_grouped.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _I64,
                                                  _I64, _INT, _INT, _F, _P, _P]
    lib.oracle_route_sigmoid_grouped.restype = _I64
    lib.oracle_dispatch.argtypes = [_P, _I64, _I64, _I64, _P, _P, _P, _P]
    lib.oracle_dispatch.restype = _I64
    lib.oracle_gather.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _P]
    lib.oracle_gather.restype = None
    lib.oracle_swiglu_rows.argtypes = [_P, _INT, _I64, _P, _P, _P, _P, _I64,
                                       _I64, _I64, _P]
    lib.oracle_swiglu_rows.restype = _INT
    lib.oracle_experts_dispatched.argtypes = [_P, _INT, _P, _I64, _P, _P, _P,
                                              _I64, _I64, _P]
    lib.oracle_experts_dispatched.restype = _INT
    lib.oracle_combine.argtypes = [_P, _INT, _P, _INT, _P, _I64, _I64, _I64, _P]
    lib.oracle_combine.restype = None
    lib.oracle_combine_v2.argtypes = [_P, _INT, _P, _INT, _P, _P, _I64, _I64, _I64, _I64,
                                      _P, _P, _P, _P, _P, _P, _INT, _INT, _I64, _I64, _I64, _P]
    lib.oracle_combine_v2.restype = _INT
    lib.oracle_rmsnorm.argtypes = [_P, _INT, _P, _INT, _F, _I64, _I64, _P,
                                   _INT, _P]
    lib.oracle_rmsnorm.restype = _INT
    lib.oracle_add_rmsnorm.argtypes = [_P, _P, _INT, _P, _INT, _F, _I64, _I64,
                                       _P, _P, _P]
    lib.oracle_add_rmsnorm.restype = _INT
    _D = ctypes.c_double
    lib.oracle_router_weights.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _INT, _INT, _D,
                                          _P, _INT]
    lib.oracle_router_weights.restype = _I64
    lib.oracle_router_backward.argtypes = [_P, _INT, _I64, _I64, _P, _I64, _P, _INT, _INT,
                                           _INT, _D, _P, _INT]
    lib.oracle_router_backward.restype = _I64
    lib.oracle_combine_backward.argtypes = [_P, _INT, _P, _INT, _P, _P, _INT, _I64, _I64,
                                            _I64, _I64, _P, _P]
    lib.oracle_combine_backward.restype = None
    lib.oracle_swiglu_backward_rows.argtypes = [_P, _INT, _I64, _P, _P, _P, _P, _I64, _I64,
                                                _I64, _P, _INT, _P, _P, _P, _P]
    lib.oracle_swiglu_backward_rows.restype = _INT
    lib.oracle_swiglu_cache_rows.argtypes = [_P, _INT, _I64, _P, _P, _P, _I64, _I64, _I64,
                                             _P, _P, _P]
    lib.oracle_swiglu_cache_rows.restype = _INT
    lib.oracle_dispatch_backward.argtypes = [_P, _INT, _P, _I64, _I64, _I64, _P]
    lib.oracle_dispatch_backward.restype = None
    return lib


def _storage(dt: str):
    return {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16,
            "f64": np.float64}[dt]


def _arr(a, dt: str):
    """Contiguous array in the storage type of dtype ``dt``."""
    a = np.asarray(a)
    if dt == "f16" and a.dtype == np.float16:
        a = a.view(np.uint16)
    want = _storage(dt)
    if a.dtype != want:
        raise TypeError(f"dtype {dt} wants {np.dtype(want)} storage, got {a.dtype}")
    return np.ascontiguousarray(a)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_index(ix, n: int, what: str, allow_negative: bool = False):
    """Raise ValueError unless every entry of ``ix`` indexes one of ``n`` rows
    (entries < 0 mean "no row" where ``allow_negative``). The C routines
    trust their index arrays; this keeps a malformed one (an oracle mutant's
    offsets, say) from reading or writing outside a buffer."""
    ix = np.asarray(ix)
    if ix.size == 0:
        return
    lo = ix.min()
    if ix.max() >= n or (lo < 0 and not allow_negative):
        raise ValueError(f"{what}: index outside [0, {n})")


def _check_offsets(offsets, rows: int, what: str):
    """Segment offsets [E+1]: non-decreasing from 0 and within ``rows`` rows."""
    o = np.asarray(offsets, dtype=np.int64)
    if o.size == 0 or o[0] != 0 or np.any(np.diff(o) < 0) or o[-1] > rows:
        raise ValueError(f"{what}: offsets not a partition of at most {rows} rows")


def convert(a, src_dt: str, dst_dt: str, lib=None):
    """Element-wise dtype conversion (exact upcast, RNE downcast)."""
    lib = lib or load_library()
    a = _arr(a, src_dt)
    out = np.empty(a.shape, dtype=_storage(dst_dt))
    lib.oracle_convert(_ptr(a), DTYPE_CODES[src_dt], _ptr(out),
                       DTYPE_CODES[dst_dt], a.size)
    return out


def to_f64(a, dt: str, lib=None):
    return convert(a, dt, "f64", lib)


def route(logits, ldt: str, top_k: int, renormalize: bool, lib=None):
    """Softmax top-k routing (ruDNN user guide, section 4 "Routing contract").

    Returns ``(idx uint32 [T,k], w [T,k] in ldt storage, invalid_rows)``.
    """
    lib = lib or load_library()
    logits = _arr(logits, ldt)
    T, E = logits.shape
    idx = np.empty((T, top_k), dtype=np.uint32)
    w = np.empty((T, top_k), dtype=_storage(ldt))
    n = lib.oracle_route(_ptr(logits), DTYPE_CODES[ldt], T, E, top_k,
                         int(bool(renormalize)), _ptr(idx), _ptr(w))
    if n < 0:
        raise ValueError("oracle_route: bad arguments")
    return idx, w, int(n)


def route_sigmoid_grouped(logits, ldt: str, bias, top_k: int, groups: int,
                          selected_groups: int, group_top_two: bool, renormalize: bool,
                          scale: float, lib=None):
    """Group-limited sigmoid routing (ruDNN user guide, section 10).

    ``bias`` is a float32 ``[E]`` correction or None. Returns ``(idx uint32
    [T,k], w [T,k] in ldt storage, invalid_rows)``.
    """
    lib = lib or load_library()
    logits = _arr(logits, ldt)
    T, E = logits.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if b is not None and b.shape != (E,):
        raise ValueError("bias must have shape [E]")
    idx = np.empty((T, top_k), dtype=np.uint32)
    w = np.empty((T, top_k), dtype=_storage(ldt))
    n = lib.oracle_route_sigmoid_grouped(
        _ptr(logits), DTYPE_CODES[ldt], T, E, None if b is None else _ptr(b), top_k, groups,
        selected_groups, int(bool(group_top_two)), int(bool(renormalize)), float(scale),
        _ptr(idx), _ptr(w))
    if n < 0:
        raise ValueError("oracle_route_sigmoid_grouped: arguments outside the limits")
    return idx, w, int(n)


def dispatch(idx, E: int, lib=None):
    """Compact no-drop dispatch (ruDNN user guide, section 5).

    Returns ``(counts [E], offsets [E+1], row_of [T*k], src_of [T*k], bad)``
    as int32 arrays; ``bad`` counts indices >= E (they get ``row_of = -1``).
    """
    lib = lib or load_library()
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    row_of = np.empty(T * k, dtype=np.int32)
    src_of = np.empty(T * k, dtype=np.int32)
    bad = lib.oracle_dispatch(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets),
                              _ptr(row_of), _ptr(src_of))
    if bad < 0:
        raise ValueError("oracle_dispatch: bad arguments")
    return counts, offsets, row_of, src_of, int(bad)


def gather(x, dt: str, top_k: int, src_of, rows: int, lib=None):
    """``x_disp[r] = x[src_of[r] // top_k]`` for the first ``rows`` rows."""
    lib = lib or load_library()
    x = _arr(x, dt)
    H = x.shape[1]
    src_of = np.ascontiguousarray(src_of, dtype=np.int32)
    if src_of.size < rows:
        raise ValueError("gather: fewer src_of entries than rows")
    _check_index(src_of[:rows] // top_k, x.shape[0], "gather")
    out = np.zeros((rows, H), dtype=_storage(dt))
    lib.oracle_gather(_ptr(x), DTYPE_CODES[dt], H, top_k, _ptr(src_of), rows,
                      _ptr(out))
    return out


def swiglu_rows(xrows, dt: str, expert_of_row, gate, up, down, lib=None):
    """Bias-free SwiGLU expert FFN on a list of (row, expert) pairs, in double.

    ``gate``/``up`` are ``[E,I,H]``, ``down`` is ``[E,H,I]``, all in ``dt``.
    """
    lib = lib or load_library()
    xrows = _arr(xrows, dt)
    gate, up, down = _arr(gate, dt), _arr(up, dt), _arr(down, dt)
    E, I, H = gate.shape
    n = xrows.shape[0]
    eor = np.ascontiguousarray(expert_of_row, dtype=np.int32)
    if eor.size != n:
        raise ValueError("swiglu_rows: one expert id per row")
    out = np.empty((n, H), dtype=np.float64)
    rc = lib.oracle_swiglu_rows(_ptr(xrows), DTYPE_CODES[dt], n, _ptr(eor),
                                _ptr(gate), _ptr(up), _ptr(down), E, H, I,
                                _ptr(out))
    if rc != 0:
        raise ValueError("oracle_swiglu_rows: expert id out of range")
    return out


def experts_dispatched(x_disp, dt: str, offsets, gate, up, down, lib=None):
    """SwiGLU experts on dispatched rows; rows of expert e are
    ``[offsets[e], offsets[e+1])``. Returns ``[offsets[E], H]`` float64."""
    lib = lib or load_library()
    x_disp = _arr(x_disp, dt)
    gate, up, down = _arr(gate, dt), _arr(up, dt), _arr(down, dt)
    E, I, H = gate.shape
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    if offsets.size != E + 1:
        raise ValueError("experts_dispatched: offsets must have E + 1 entries")
    _check_offsets(offsets, x_disp.shape[0], "experts_dispatched")
    out = np.empty((int(offsets[E]), H), dtype=np.float64)
    rc = lib.oracle_experts_dispatched(_ptr(x_disp), DTYPE_CODES[dt],
                                       _ptr(offsets), E, _ptr(gate), _ptr(up),
                                       _ptr(down), H, I, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_experts_dispatched failed")
    return out


def combine(out_disp, odt: str, w, wdt: str, row_of, top_k: int, lib=None):
    """Weighted combine back to token order, in double (slot order)."""
    lib = lib or load_library()
    out_disp = _arr(out_disp, odt)
    w = _arr(w, wdt)
    row_of = np.ascontiguousarray(row_of, dtype=np.int32)
    T = row_of.size // top_k
    H = out_disp.shape[1]
    _check_index(row_of, out_disp.shape[0], "combine", allow_negative=True)
    if w.size < T * top_k:
        raise ValueError("combine: fewer weights than slots")
    y = np.empty((T, H), dtype=np.float64)
    lib.oracle_combine(_ptr(out_disp), DTYPE_CODES[odt], _ptr(w),
                       DTYPE_CODES[wdt], _ptr(row_of), T, top_k, H, _ptr(y))
    return y


def combine_v2(out_disp, odt: str, w, wdt: str, row_of, top_k: int, xdt: str, ids=None,
               E: int = 0, zero: int = 0, copy: int = 0, const: int = 0, ori_x=None,
               alpha1=None, alpha2=None, const_v=None, shared_x=None, mask=None, lib=None):
    """Combine of aclnnMoeDistributeCombineAddRmsNormV2 (special experts,
    shared expert, active mask). ``mask`` is None, bool [T] or bool [T, k];
    ``ori_x``, ``alpha1``, ``alpha2``, ``const_v``, ``shared_x`` in ``xdt``
    storage. Returns the unrounded float64 ``[T, H]``."""
    lib = lib or load_library()
    out_disp = _arr(out_disp, odt)
    w = _arr(w, wdt)
    T = w.shape[0]
    H = out_disp.shape[1]
    row_of = np.ascontiguousarray(row_of, dtype=np.int32)
    _check_index(row_of, out_disp.shape[0], "combine_v2", allow_negative=True)
    ids_a = None if ids is None else np.ascontiguousarray(ids, dtype=np.uint32)
    opt = {n: (None if v is None else _arr(v, xdt)) for n, v in
           dict(ori_x=ori_x, alpha1=alpha1, alpha2=alpha2, const_v=const_v,
                shared_x=shared_x).items()}
    mask_a = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    mdims = 0 if mask_a is None else mask_a.ndim
    y = np.empty((T, H), dtype=np.float64)
    p = lambda a: None if a is None else _ptr(a)
    rc = lib.oracle_combine_v2(_ptr(out_disp), DTYPE_CODES[odt], _ptr(w), DTYPE_CODES[wdt],
                               _ptr(row_of), p(ids_a), E, zero, copy, const, p(opt["ori_x"]),
                               p(opt["alpha1"]), p(opt["alpha2"]), p(opt["const_v"]),
                               p(opt["shared_x"]), p(mask_a), mdims, DTYPE_CODES[xdt], T,
                               top_k, H, _ptr(y))
    if rc == -2:
        raise ValueError("oracle_combine_v2: a 1-D active mask must keep its tokens first")
    if rc != 0:
        raise ValueError("oracle_combine_v2: missing inputs for the configured experts or mask")
    return y


def rmsnorm(x, dt: str, gamma, gdt: str, eps: float, out_dt: str | None = None,
            lib=None):
    """Last-axis RMSNorm (ruDNN user guide, section 7). Returns (y, rstd)."""
    lib = lib or load_library()
    out_dt = out_dt or dt
    x = _arr(x, dt)
    gamma = _arr(gamma, gdt)
    T, H = x.shape
    y = np.empty((T, H), dtype=_storage(out_dt))
    rstd = np.empty(T, dtype=np.float32)
    rc = lib.oracle_rmsnorm(_ptr(x), DTYPE_CODES[dt], _ptr(gamma),
                            DTYPE_CODES[gdt], float(eps), T, H, _ptr(y),
                            DTYPE_CODES[out_dt], _ptr(rstd))
    if rc != 0:
        raise ValueError("oracle_rmsnorm: eps must be finite and > 0")
    return y, rstd


def add_rmsnorm(combine_f64, residual, rdt: str, gamma, gdt: str, eps: float,
                lib=None):
    """Residual Add + RMSNorm (aclnnMoeDistributeCombineAddRmsNormV2 formula).

    Returns ``(y, x_out, rstd)``; y and x_out in the residual dtype.
    """
    lib = lib or load_library()
    comb = np.ascontiguousarray(combine_f64, dtype=np.float64)
    residual = _arr(residual, rdt)
    gamma = _arr(gamma, gdt)
    T, H = residual.shape
    y = np.empty((T, H), dtype=_storage(rdt))
    x_out = np.empty((T, H), dtype=_storage(rdt))
    rstd = np.empty(T, dtype=np.float32)
    rc = lib.oracle_add_rmsnorm(_ptr(comb), _ptr(residual), DTYPE_CODES[rdt],
                                _ptr(gamma), DTYPE_CODES[gdt], float(eps), T, H,
                                _ptr(y), _ptr(x_out), _ptr(rstd))
    if rc != 0:
        raise ValueError("oracle_add_rmsnorm: eps must be finite and > 0")
    return y, x_out, rstd


def forward(x, dt: str, logits, ldt: str, gate, up, down, top_k: int,
            renormalize: bool, lib=None):
    """The whole local chain (ruDNN user guide, sections 3 and 6): route,
    dispatch, SwiGLU experts, combine. Returns a dict of every stage; ``y``
    is the unrounded float64 output ``[T, H]``."""
    lib = lib or load_library()
    idx, w, invalid = route(logits, ldt, top_k, renormalize, lib)
    return _forward_routed(x, dt, idx, w, ldt, invalid, gate, up, down, lib)


def forward_sigmoid_grouped(x, dt: str, logits, ldt: str, bias, gate, up, down, top_k: int,
                            groups: int, selected_groups: int, group_top_two: bool,
                            renormalize: bool, scale: float, lib=None):
    """The same chain with group-limited sigmoid routing (ruDNN user guide,
    section 10, forward_sigmoid_grouped)."""
    lib = lib or load_library()
    idx, w, invalid = route_sigmoid_grouped(logits, ldt, bias, top_k, groups, selected_groups,
                                            group_top_two, renormalize, scale, lib)
    return _forward_routed(x, dt, idx, w, ldt, invalid, gate, up, down, lib)


def _forward_routed(x, dt, idx, w, ldt, invalid, gate, up, down, lib):
    top_k = idx.shape[1]
    E = np.asarray(gate).shape[0]
    counts, offsets, row_of, src_of, bad = dispatch(idx, E, lib)
    rows = int(offsets[E])
    x_disp = gather(x, dt, top_k, src_of, rows, lib)
    out_disp = experts_dispatched(x_disp, dt, offsets, gate, up, down, lib)
    y = combine(out_disp, "f64", w, ldt, row_of, top_k, lib)
    return {"idx": idx, "w": w, "invalid_rows": invalid, "counts": counts,
            "offsets": offsets, "row_of": row_of, "src_of": src_of,
            "x_disp": x_disp, "out_disp": out_disp, "y": y}


def forward_tokens(tokens, x, dt: str, logits, ldt: str, gate, up, down,
                   top_k: int, renormalize: bool, lib=None, sigmoid_grouped=None):
    """The same chain evaluated for a subset of tokens only (used to sample
    full-size workloads). A token's output depends only on its own row of x
    and logits, so this equals rows ``tokens`` of :func:`forward`. With
    ``sigmoid_grouped`` a dict of :func:`route_sigmoid_grouped`'s arguments
    (bias, groups, selected_groups, group_top_two, scale), the tokens are
    routed that way instead. Returns ``(idx, w, y)`` for those tokens."""
    lib = lib or load_library()
    tokens = np.asarray(tokens, dtype=np.int64)
    lg = _arr(logits, ldt)[tokens]
    xs = _arr(x, dt)[tokens]
    if sigmoid_grouped is None:
        idx, w, _ = route(lg, ldt, top_k, renormalize, lib)
    else:
        sg = sigmoid_grouped
        idx, w, _ = route_sigmoid_grouped(lg, ldt, sg["bias"], top_k, sg["groups"],
                                          sg["selected_groups"], sg["group_top_two"],
                                          renormalize, sg["scale"], lib)
    n = tokens.size
    rows = np.repeat(xs, top_k, axis=0)
    out = swiglu_rows(rows, dt, idx.reshape(-1).astype(np.int32), gate, up,
                      down, lib)
    row_of = np.arange(n * top_k, dtype=np.int32)
    y = combine(out, "f64", w, ldt, row_of, top_k, lib)
    return idx, w, y


# ---- first-order training (ruDNN user guide, section 12) -----------------

SCORING = {"softmax": 0, "sigmoid": 1}


def _idx64(idx):
    """Selection indices as int64 (U32, I32 and I64 are all accepted)."""
    a = np.asarray(idx)
    if a.dtype == np.uint32 or a.dtype == np.uint64:
        a = a.astype(np.uint64)
        a = np.where(a > np.uint64(2**62), np.uint64(2**62), a).astype(np.int64)
    return np.ascontiguousarray(a, dtype=np.int64)


def router_weights(logits, ldt: str, idx, scoring: str = "softmax",
                   renormalize: bool = False, scale: float = 1.0, out_dt: str = "f32",
                   lib=None):
    """Weights of a fixed selection (selected_router_weights). Returns
    ``(w [T,k] in out_dt storage, nan_rows)``."""
    lib = lib or load_library()
    logits = _arr(logits, ldt)
    T, E = logits.shape
    idx = _idx64(idx)
    k = idx.shape[1]
    w = np.empty((T, k), dtype=_storage(out_dt))
    n = lib.oracle_router_weights(_ptr(logits), DTYPE_CODES[ldt], T, E, _ptr(idx), k,
                                  SCORING[scoring], int(bool(renormalize)), float(scale),
                                  _ptr(w), DTYPE_CODES[out_dt])
    if n < 0:
        raise ValueError("oracle_router_weights: bad arguments")
    return w, int(n)


def router_backward(logits, ldt: str, idx, grad_w, gwdt: str = "f32",
                    scoring: str = "softmax", renormalize: bool = False, scale: float = 1.0,
                    out_dt: str | None = None, lib=None):
    """Logits gradient of :func:`router_weights` (selected_router_backward).
    Returns ``(dlogits [T,E] in out_dt storage (default the logits dtype),
    nan_rows)``."""
    lib = lib or load_library()
    out_dt = out_dt or ldt
    logits = _arr(logits, ldt)
    T, E = logits.shape
    idx = _idx64(idx)
    k = idx.shape[1]
    gw = _arr(grad_w, gwdt)
    dl = np.empty((T, E), dtype=_storage(out_dt))
    n = lib.oracle_router_backward(_ptr(logits), DTYPE_CODES[ldt], T, E, _ptr(idx), k,
                                   _ptr(gw), DTYPE_CODES[gwdt], SCORING[scoring],
                                   int(bool(renormalize)), float(scale), _ptr(dl),
                                   DTYPE_CODES[out_dt])
    if n < 0:
        raise ValueError("oracle_router_backward: bad arguments")
    return dl, int(n)


def combine_backward(out_disp, odt: str, w, wdt: str, row_of, grad_y, gdt: str, top_k: int,
                     lib=None):
    """Backward of the weighted combine. Returns float64 ``(dexpert [rows,H],
    dw [T,k])``."""
    lib = lib or load_library()
    out_disp = _arr(out_disp, odt)
    w = _arr(w, wdt)
    gy = _arr(grad_y, gdt)
    row_of = np.ascontiguousarray(row_of, dtype=np.int32)
    T, H = gy.shape
    rows = out_disp.shape[0]
    _check_index(row_of, rows, "combine_backward", allow_negative=True)
    if row_of.size != T * top_k or w.size < T * top_k:
        raise ValueError("combine_backward: row_of / weights do not match [T, top_k]")
    dexp = np.empty((rows, H), dtype=np.float64)
    dw = np.empty((T, top_k), dtype=np.float64)
    lib.oracle_combine_backward(_ptr(out_disp), DTYPE_CODES[odt], _ptr(w), DTYPE_CODES[wdt],
                                _ptr(row_of), _ptr(gy), DTYPE_CODES[gdt], T, top_k, H, rows,
                                _ptr(dexp), _ptr(dw))
    return dexp, dw


def swiglu_backward_rows(xrows, dt: str, expert_of_row, gate, up, down, dout, ddt: str,
                         lib=None):
    """Backward of the SwiGLU experts on (row, expert) pairs, in double.
    Returns ``(dx [n,H], dgate [E,I,H], dup [E,I,H], ddown [E,H,I])``."""
    lib = lib or load_library()
    xrows = _arr(xrows, dt)
    gate, up, down = _arr(gate, dt), _arr(up, dt), _arr(down, dt)
    dout = _arr(dout, ddt)
    E, I, H = gate.shape
    n = xrows.shape[0]
    eor = np.ascontiguousarray(expert_of_row, dtype=np.int32)
    if eor.size != n or dout.shape[0] != n:
        raise ValueError("swiglu_backward_rows: one expert id and one output gradient per row")
    dx = np.empty((n, H), dtype=np.float64)
    dg = np.empty((E, I, H), dtype=np.float64)
    du = np.empty((E, I, H), dtype=np.float64)
    dd = np.empty((E, H, I), dtype=np.float64)
    rc = lib.oracle_swiglu_backward_rows(_ptr(xrows), DTYPE_CODES[dt], n, _ptr(eor),
                                         _ptr(gate), _ptr(up), _ptr(down), E, H, I,
                                         _ptr(dout), DTYPE_CODES[ddt], _ptr(dx), _ptr(dg),
                                         _ptr(du), _ptr(dd))
    if rc != 0:
        raise ValueError("oracle_swiglu_backward_rows: expert id out of range")
    return dx, dg, du, dd


def experts_backward_dispatched(x_disp, dt: str, offsets, gate, up, down, dout, ddt: str,
                                lib=None):
    """:func:`swiglu_backward_rows` on dispatched rows (rows of expert e are
    ``[offsets[e], offsets[e+1])``)."""
    offsets = np.asarray(offsets, dtype=np.int64)
    E = np.asarray(gate).shape[0]
    _check_offsets(offsets, np.asarray(x_disp).shape[0], "experts_backward_dispatched")
    if offsets.size != E + 1 or offsets[E] != np.asarray(x_disp).shape[0]:
        raise ValueError("experts_backward_dispatched: offsets[E] must equal the rows given")
    owner = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    return swiglu_backward_rows(x_disp, dt, owner, gate, up, down, dout, ddt, lib)


def dispatch_backward(dinput, dt: str, row_of, top_k: int, lib=None):
    """Backward of the dispatch gather: the selected rows summed back to their
    token (no routing weight). Returns float64 ``[T,H]``."""
    lib = lib or load_library()
    d = _arr(dinput, dt)
    row_of = np.ascontiguousarray(row_of, dtype=np.int32)
    T = row_of.size // top_k
    H = d.shape[1]
    _check_index(row_of, d.shape[0], "dispatch_backward", allow_negative=True)
    dx = np.empty((T, H), dtype=np.float64)
    lib.oracle_dispatch_backward(_ptr(d), DTYPE_CODES[dt], _ptr(row_of), T, top_k, H,
                                 _ptr(dx))
    return dx


def experts_cache_dispatched(x_disp, dt: str, offsets, gate, up, lib=None):
    """The training forward's cache on dispatched rows: ``(g, u, h)``, each
    float64 ``[offsets[E], I]``."""
    lib = lib or load_library()
    x_disp = _arr(x_disp, dt)
    gate, up = _arr(gate, dt), _arr(up, dt)
    E, I, H = gate.shape
    offsets = np.asarray(offsets, dtype=np.int64)
    if offsets.size != E + 1:
        raise ValueError("experts_cache_dispatched: offsets must have E + 1 entries")
    _check_offsets(offsets, x_disp.shape[0], "experts_cache_dispatched")
    n = int(offsets[E])
    owner = np.ascontiguousarray(np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets)))
    g = np.empty((n, I)); u = np.empty((n, I)); h = np.empty((n, I))
    rc = lib.oracle_swiglu_cache_rows(_ptr(x_disp), DTYPE_CODES[dt], n, _ptr(owner), _ptr(gate),
                                      _ptr(up), E, H, I, _ptr(g), _ptr(u), _ptr(h))
    if rc != 0:
        raise ValueError("oracle_swiglu_cache_rows: expert id out of range")
    return g, u, h
