"""GB300-native local Mixture-of-Experts FFN forward.

A thin ctypes binding of the C ABI in ``include/moe.h``: every function here
has the name of the C entry point it calls and only marshals arguments
(torch tensors -> device pointers and sizes, the current CUDA stream). All
compute runs in the hand-written sm_103a kernels of ``_lib/libmoe_gb300.so``;
there is no fallback: if the library is missing the call raises.

Tensors must be contiguous CUDA tensors. Expert indices are U32 in the ABI;
the binding stores them in ``torch.int32`` tensors (same bits, values < 1024).
Outputs may be passed in (``out=``-style keyword arguments) to reuse memory;
otherwise they are allocated with torch on the input's device. Workspaces are
torch ``uint8`` tensors sized by the matching ``*_workspace_size`` call.

Sources: ruDNN user guide sections 3-7 (routing, dispatch, SwiGLU experts,
combine, RMSNorm), section 10 (grouped sigmoid routing) and section 12
(first-order MoE training); aclnnMoeDistributeCombineAddRmsNormV2 "Function"
formula.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_gb300.so")
LIB_PATH_DEBUG = os.path.join(_PKG, "_lib", "libmoe_gb300_debug.so")
_DEFAULT_LIB_PATH = LIB_PATH


def library_path(env=None) -> str:
    """The library the binding loads: the bounds-checking build when the
    environment variable MOE_DEBUG_BOUNDS is 1, the normal one when it is
    unset, empty or 0; any other value is an error."""
    env = os.environ if env is None else env
    flag = env.get("MOE_DEBUG_BOUNDS", "")
    if flag in ("", "0"):
        return LIB_PATH
    if flag == "1":
        return LIB_PATH_DEBUG
    raise ValueError(f"MOE_DEBUG_BOUNDS must be unset, 0 or 1, not {flag!r}")

MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
DTYPE_CODES = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16,
               torch.float16: MOE_F16}

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE",
                3: "MOE_ERR_DTYPE", 4: "MOE_ERR_VALUE", 5: "MOE_ERR_ALIGN",
                6: "MOE_ERR_WORKSPACE", 7: "MOE_ERR_CUDA",
                8: "MOE_ERR_DEVICE_TIMEOUT", 9: "MOE_ERR_BAD_INDEX", 10: "MOE_ERR_BOUNDS"}

EXPORTED = ["moe_status_string", "moe_abi_version", "moe_last_error_detail",
            "moe_route", "moe_route_sigmoid_grouped", "moe_dispatch_workspace_size",
            "moe_dispatch", "moe_dispatch_special", "moe_combine_v2", "moe_rmsnorm",
            "moe_dispatch_noalloc",
            "moe_experts_workspace_size", "moe_experts_forward", "moe_combine",
            "moe_combine_add_rmsnorm", "moe_forward_workspace_size",
            "moe_forward", "moe_forward_sigmoid_grouped", "moe_device_status",
            "moe_router_weights", "moe_router_backward", "moe_combine_backward",
            "moe_dispatch_backward", "moe_experts_training_cache_size",
            "moe_experts_forward_training", "moe_experts_backward_workspace_size",
            "moe_experts_backward", "moe_forward_workspace_size_ex", "moe_forward_ex",
            "moe_forward_workspace_layout", "moe_set_wait_limit_ns", "moe_wait_limit_ns",
            "moe_selftest_wait_expiry_workspace_size", "moe_selftest_wait_expiry"]

MOE_FORWARD_DETERMINISTIC = 1

MOE_SCORING_SOFTMAX, MOE_SCORING_SIGMOID = 0, 1
SCORING_CODES = {"softmax": MOE_SCORING_SOFTMAX, "sigmoid": MOE_SCORING_SIGMOID}
INDEX_CODES = {torch.int32: 1, torch.int64: 2}
if hasattr(torch, "uint32"):
    INDEX_CODES[torch.uint32] = 0

_lock = threading.Lock()
_lib = None

_P, _I64, _INT, _SZ, _F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                           ctypes.c_size_t, ctypes.c_float)


class CombineExtras(ctypes.Structure):
    """Mirror of ``moe_combine_extras`` (include/moe.h)."""
    _fields_ = [("expert_indices", ctypes.c_void_p), ("num_experts", ctypes.c_int64),
                ("zero_experts", ctypes.c_int64), ("copy_experts", ctypes.c_int64),
                ("const_experts", ctypes.c_int64), ("ori_x", ctypes.c_void_p),
                ("const_alpha1", ctypes.c_void_p), ("const_alpha2", ctypes.c_void_p),
                ("const_v", ctypes.c_void_p), ("shared_expert_x", ctypes.c_void_p),
                ("active_mask", ctypes.c_void_p), ("active_mask_dims", ctypes.c_int)]


class SigmoidGroupedRouting(ctypes.Structure):
    """Mirror of ``moe_sigmoid_grouped_routing`` (include/moe.h)."""
    _fields_ = [("bias", ctypes.c_void_p), ("groups", ctypes.c_int),
                ("selected_groups", ctypes.c_int), ("group_top_two", ctypes.c_int),
                ("scale", ctypes.c_float)]


class ForwardOptions(ctypes.Structure):
    """Mirror of ``moe_forward_options`` (include/moe.h)."""
    _fields_ = [("flags", ctypes.c_uint), ("sigmoid_grouped", ctypes.POINTER(SigmoidGroupedRouting)),
                ("experts_begin_event", ctypes.c_void_p), ("experts_end_event", ctypes.c_void_p)]


class ForwardLayout(ctypes.Structure):
    """Mirror of ``moe_forward_layout`` (include/moe.h)."""
    _fields_ = [(n, ctypes.c_size_t) for n in ("expert_indices", "weights", "counts", "offsets",
                                               "row_of", "src_of", "x_disp", "total")]


class MoeError(RuntimeError):
    """A non-zero status returned by the C ABI."""

    def __init__(self, code: int, fn: str, detail: str = ""):
        self.code = code
        self.name = STATUS_NAMES.get(code, str(code))
        super().__init__(f"{fn}: {self.name}" + (f" ({detail})" if detail else ""))


def _bind(lib):
    sig = {
        "moe_status_string": ([_INT], ctypes.c_char_p),
        "moe_abi_version": ([], _INT),
        "moe_last_error_detail": ([], ctypes.c_char_p),
        "moe_route": ([_P, _INT, _I64, _I64, _INT, _INT, _P, _P, _P], _INT),
        "moe_route_sigmoid_grouped": ([_P, _INT, _I64, _I64, _P, _INT, _INT, _INT, _INT,
                                       _INT, _F, _P, _P, _P], _INT),
        "moe_dispatch_workspace_size": ([_I64, _INT, _I64], _SZ),
        "moe_dispatch": ([_P, _I64, _INT, _I64, _P, _INT, _I64, _P, _P, _P, _P,
                          _P, _P, _SZ, _P], _INT),
        "moe_dispatch_noalloc": ([_P, _I64, _INT, _I64, _P, _INT, _I64, _P, _P, _P,
                                  _P, _P, _P], _INT),
        "moe_dispatch_special": ([_P, _I64, _INT, _I64, _I64, _P, _INT, _I64, _P, _P, _P,
                                  _P, _P, _P, _SZ, _P], _INT),
        "moe_combine_v2": ([_P, _INT, _P, _INT, _P, ctypes.POINTER(CombineExtras), _P, _P,
                            _INT, _F, _I64, _INT, _I64, _P, _INT, _P, _P, _P], _INT),
        "moe_rmsnorm": ([_P, _INT, _P, _INT, _F, _I64, _I64, _P, _P, _P], _INT),
        "moe_experts_workspace_size": ([_I64, _I64, _I64, _I64, _INT], _SZ),
        "moe_experts_forward": ([_P, _P, _I64, _P, _P, _P, _I64, _I64, _I64,
                                 _INT, _P, _INT, _P, _SZ, _P], _INT),
        "moe_combine": ([_P, _INT, _P, _INT, _P, _I64, _INT, _I64, _P, _INT, _P], _INT),
        "moe_combine_add_rmsnorm": ([_P, _INT, _P, _INT, _P, _P, _INT, _P, _INT,
                                     _F, _I64, _INT, _I64, _P, _P, _P, _P], _INT),
        "moe_forward_workspace_size": ([_I64, _I64, _I64, _I64, _INT, _INT,
                                        _INT], _SZ),
        "moe_forward": ([_P, _INT, _P, _INT, _P, _P, _P, _I64, _I64, _I64, _I64,
                         _INT, _INT, _P, _P, _SZ, _P], _INT),
        "moe_forward_sigmoid_grouped": ([_P, _INT, _P, _INT, _P, _P, _P, _P, _I64, _I64,
                                         _I64, _I64, _INT, _INT, _INT, _INT, _INT, _F, _P,
                                         _P, _SZ, _P], _INT),
        "moe_device_status": ([_P, _INT], _INT),
        "moe_router_weights": ([_P, _INT, _I64, _I64, _P, _INT, _INT, _INT, _INT, _F, _P,
                                _P], _INT),
        "moe_router_backward": ([_P, _INT, _I64, _I64, _P, _INT, _INT, _P, _INT, _INT, _F,
                                 _P, _P], _INT),
        "moe_combine_backward": ([_P, _INT, _P, _INT, _P, _P, _I64, _INT, _I64, _INT, _P, _P,
                                  _P], _INT),
        "moe_dispatch_backward": ([_P, _INT, _P, _I64, _INT, _I64, _P, _P], _INT),
        "moe_experts_training_cache_size": ([_I64, _I64, _INT], _SZ),
        "moe_experts_forward_training": ([_P, _P, _I64, _P, _P, _P, _I64, _I64, _I64, _INT,
                                          _P, _INT, _P, _SZ, _P], _INT),
        "moe_experts_backward_workspace_size": ([_I64, _I64, _I64, _I64, _INT], _SZ),
        "moe_experts_backward": ([_P, _P, _I64, _P, _P, _P, _I64, _I64, _I64, _INT, _P, _P,
                                  _P, _P, _P, _P, _P, _SZ, _P], _INT),
        "moe_forward_workspace_size_ex": ([_I64, _I64, _I64, _I64, _INT, _INT, _INT,
                                           ctypes.c_uint], _SZ),
        "moe_forward_ex": ([_P, _INT, _P, _INT, _P, _P, _P, _I64, _I64, _I64, _I64, _INT, _INT,
                            _P, _P, _SZ, ctypes.POINTER(ForwardOptions), _P], _INT),
        "moe_forward_workspace_layout": ([_I64, _I64, _I64, _I64, _INT, _INT, _INT,
                                          ctypes.c_uint, ctypes.POINTER(ForwardLayout)], _INT),
        "moe_set_wait_limit_ns": ([ctypes.c_uint64], _INT),
        "moe_wait_limit_ns": ([], ctypes.c_uint64),
        "moe_selftest_wait_expiry_workspace_size": ([_I64, _I64, _I64, _I64], _SZ),
        "moe_selftest_wait_expiry": ([_I64, _I64, _I64, _I64, _P, _P, _SZ, _P], _INT),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


def load_library(path: str | None = None):
    """Load the extension. Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            # a LIB_PATH reassigned by the caller wins over the environment
            p = path or (LIB_PATH if LIB_PATH != _DEFAULT_LIB_PATH else library_path())
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA extension not built: {p} is missing; run "
                    "mixture_experts_ffn_topk_gb300.build.build()")
            lib = _bind(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
    return _lib


def _check(rc: int, fn: str):
    if rc != 0:
        detail = load_library().moe_last_error_detail().decode(errors="replace")
        raise MoeError(rc, fn, detail)


def _code(dtype: torch.dtype) -> int:
    if dtype not in DTYPE_CODES:
        raise TypeError(f"unsupported dtype {dtype}; use float32, bfloat16 or float16")
    return DTYPE_CODES[dtype]


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(None)
    if not t.is_cuda:
        raise ValueError("tensors passed to the C ABI must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the C ABI must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _workspace(nbytes: int, device, given: torch.Tensor | None) -> torch.Tensor | None:
    if given is not None:
        return given
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _nbytes(t: torch.Tensor | None) -> int:
    return 0 if t is None else t.numel() * t.element_size()


# ----------------------------------------------------------------- entry points

def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return load_library().moe_abi_version()


def moe_route(logits: torch.Tensor, top_k: int, renormalize: bool,
              expert_indices: torch.Tensor | None = None,
              weights: torch.Tensor | None = None, stream=None):
    """Softmax top-k routing. Returns ``(expert_indices int32 [T,k],
    weights [T,k] in logits.dtype)``."""
    T, E = logits.shape
    dev = logits.device
    if expert_indices is None:
        expert_indices = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, top_k), dtype=logits.dtype, device=dev)
    rc = load_library().moe_route(_ptr(logits), _code(logits.dtype), T, E,
                                  int(top_k), int(bool(renormalize)),
                                  _ptr(expert_indices), _ptr(weights),
                                  _stream(stream))
    _check(rc, "moe_route")
    return expert_indices, weights


def moe_route_sigmoid_grouped(logits: torch.Tensor, bias: torch.Tensor | None, top_k: int,
                              groups: int, selected_groups: int, group_top_two: bool,
                              renormalize: bool, scale: float = 1.0,
                              expert_indices: torch.Tensor | None = None,
                              weights: torch.Tensor | None = None, stream=None):
    """Group-limited sigmoid routing; ``bias`` is an FP32 ``[E]`` correction
    or None. Returns ``(expert_indices int32 [T,k], weights [T,k] in
    logits.dtype)``."""
    T, E = logits.shape
    dev = logits.device
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (E,)):
        raise ValueError("bias must be float32 of shape [E]")
    if expert_indices is None:
        expert_indices = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, top_k), dtype=logits.dtype, device=dev)
    rc = load_library().moe_route_sigmoid_grouped(
        _ptr(logits), _code(logits.dtype), T, E, None if bias is None else _ptr(bias),
        int(top_k), int(groups), int(selected_groups), int(bool(group_top_two)),
        int(bool(renormalize)), float(scale), _ptr(expert_indices), _ptr(weights),
        _stream(stream))
    _check(rc, "moe_route_sigmoid_grouped")
    return expert_indices, weights


def moe_dispatch_workspace_size(T: int, top_k: int, E: int) -> int:
    return int(load_library().moe_dispatch_workspace_size(T, top_k, E))


def moe_dispatch(expert_indices: torch.Tensor, x: torch.Tensor, E: int,
                 counts=None, offsets=None, row_of=None, src_of=None,
                 x_disp=None, workspace=None, stream=None) -> dict:
    """Compact no-drop dispatch. Returns a dict with ``counts [E]``,
    ``offsets [E+1]``, ``row_of [T*k]``, ``src_of [T*k]`` (int32) and
    ``x_disp [T*k, H]``."""
    T, k = expert_indices.shape
    H = x.shape[1]
    dev = x.device
    A = T * k
    counts = counts if counts is not None else torch.empty(E, dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = row_of if row_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    src_of = src_of if src_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    x_disp = x_disp if x_disp is not None else torch.empty((A, H), dtype=x.dtype, device=dev)
    ws = _workspace(moe_dispatch_workspace_size(T, k, E), dev, workspace)
    rc = load_library().moe_dispatch(
        _ptr(expert_indices), T, k, E, _ptr(x), _code(x.dtype), H, _ptr(counts),
        _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(x_disp), _ptr(ws),
        _nbytes(ws), _stream(stream))
    _check(rc, "moe_dispatch")
    return {"counts": counts, "offsets": offsets, "row_of": row_of,
            "src_of": src_of, "x_disp": x_disp}


def moe_dispatch_special(expert_indices: torch.Tensor, x: torch.Tensor, E: int,
                         special_experts: int, counts=None, offsets=None, row_of=None,
                         src_of=None, x_disp=None, workspace=None, stream=None) -> dict:
    """:func:`moe_dispatch` where ids in ``[E, E + special_experts)`` name
    special experts: no dispatched row, not a bad index."""
    T, k = expert_indices.shape
    H = x.shape[1]
    dev = x.device
    A = T * k
    counts = counts if counts is not None else torch.empty(E, dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = row_of if row_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    src_of = src_of if src_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    x_disp = x_disp if x_disp is not None else torch.empty((A, H), dtype=x.dtype, device=dev)
    ws = _workspace(moe_dispatch_workspace_size(T, k, E), dev, workspace)
    rc = load_library().moe_dispatch_special(
        _ptr(expert_indices), T, k, E, int(special_experts), _ptr(x), _code(x.dtype), H,
        _ptr(counts), _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(x_disp), _ptr(ws),
        _nbytes(ws), _stream(stream))
    _check(rc, "moe_dispatch_special")
    return {"counts": counts, "offsets": offsets, "row_of": row_of,
            "src_of": src_of, "x_disp": x_disp}


def moe_dispatch_noalloc(expert_indices: torch.Tensor, x: torch.Tensor, E: int,
                         counts=None, offsets=None, row_of=None, src_of=None,
                         x_disp=None, stream=None) -> dict:
    """``moe_dispatch`` without a workspace, for callers that cannot allocate
    device scratch: the library keeps the scratch in a fixed 256 KiB array per
    device (see ``include/moe.h``). Same outputs as :func:`moe_dispatch`."""
    T, k = expert_indices.shape
    H = x.shape[1]
    dev = x.device
    A = T * k
    counts = counts if counts is not None else torch.empty(E, dtype=torch.int32, device=dev)
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = row_of if row_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    src_of = src_of if src_of is not None else torch.empty(A, dtype=torch.int32, device=dev)
    x_disp = x_disp if x_disp is not None else torch.empty((A, H), dtype=x.dtype, device=dev)
    rc = load_library().moe_dispatch_noalloc(
        _ptr(expert_indices), T, k, E, _ptr(x), _code(x.dtype), H, _ptr(counts),
        _ptr(offsets), _ptr(row_of), _ptr(src_of), _ptr(x_disp), _stream(stream))
    _check(rc, "moe_dispatch_noalloc")
    return {"counts": counts, "offsets": offsets, "row_of": row_of,
            "src_of": src_of, "x_disp": x_disp}


def moe_experts_workspace_size(rows: int, E: int, H: int, I: int,
                               dtype: torch.dtype) -> int:
    return int(load_library().moe_experts_workspace_size(rows, E, H, I, _code(dtype)))


def moe_experts_forward(x_disp: torch.Tensor, offsets: torch.Tensor,
                        gate: torch.Tensor, up: torch.Tensor,
                        down: torch.Tensor, out_disp=None, workspace=None,
                        out_dtype: torch.dtype | None = None,
                        stream=None) -> torch.Tensor:
    """Bias-free SwiGLU experts on dispatched rows; returns ``out_disp`` in
    ``out_dtype`` (default: the activation dtype; ``torch.float32`` keeps the
    expert outputs unrounded)."""
    rows, H = x_disp.shape
    E, I, _ = gate.shape
    dev = x_disp.device
    if out_disp is not None:
        out_dtype = out_disp.dtype
    out_dtype = out_dtype or x_disp.dtype
    if out_disp is None:
        out_disp = torch.empty((rows, H), dtype=out_dtype, device=dev)
    ws = _workspace(moe_experts_workspace_size(rows, E, H, I, x_disp.dtype), dev, workspace)
    rc = load_library().moe_experts_forward(
        _ptr(x_disp), _ptr(offsets), rows, _ptr(gate), _ptr(up), _ptr(down), E,
        H, I, _code(x_disp.dtype), _ptr(out_disp), _code(out_dtype), _ptr(ws),
        _nbytes(ws), _stream(stream))
    _check(rc, "moe_experts_forward")
    return out_disp


def moe_combine(out_disp: torch.Tensor, weights: torch.Tensor,
                row_of: torch.Tensor, y=None, dtype: torch.dtype | None = None,
                stream=None) -> torch.Tensor:
    """Weighted combine back to token order; returns ``y [T, H]`` in
    ``dtype`` (default: ``y.dtype`` if given, else ``out_disp.dtype``)."""
    T, k = weights.shape
    H = out_disp.shape[1]
    if y is not None:
        dtype = y.dtype
    dtype = dtype or out_disp.dtype
    if y is None:
        y = torch.empty((T, H), dtype=dtype, device=out_disp.device)
    rc = load_library().moe_combine(
        _ptr(out_disp), _code(out_disp.dtype), _ptr(weights),
        _code(weights.dtype), _ptr(row_of), T, k, H, _ptr(y), _code(dtype),
        _stream(stream))
    _check(rc, "moe_combine")
    return y


def moe_combine_add_rmsnorm(out_disp: torch.Tensor, weights: torch.Tensor,
                            row_of: torch.Tensor, residual: torch.Tensor,
                            gamma: torch.Tensor, eps: float, y=None,
                            x_out=None, rstd=None, stream=None):
    """Combine + residual Add + RMSNorm; returns ``(y, x_out, rstd)`` with y
    and x_out in ``residual.dtype``."""
    T, k = weights.shape
    H = out_disp.shape[1]
    dev = out_disp.device
    dt = residual.dtype
    y = y if y is not None else torch.empty((T, H), dtype=dt, device=dev)
    x_out = x_out if x_out is not None else torch.empty((T, H), dtype=dt, device=dev)
    rstd = rstd if rstd is not None else torch.empty(T, dtype=torch.float32, device=dev)
    rc = load_library().moe_combine_add_rmsnorm(
        _ptr(out_disp), _code(out_disp.dtype), _ptr(weights),
        _code(weights.dtype), _ptr(row_of), _ptr(residual), _code(dt), _ptr(gamma),
        _code(gamma.dtype), float(eps), T, k, H, _ptr(y), _ptr(x_out),
        _ptr(rstd), _stream(stream))
    _check(rc, "moe_combine_add_rmsnorm")
    return y, x_out, rstd


def moe_combine_v2(out_disp: torch.Tensor, weights: torch.Tensor, row_of: torch.Tensor,
                   dtype: torch.dtype, expert_indices=None, num_experts: int = 1,
                   zero_experts: int = 0, copy_experts: int = 0, const_experts: int = 0,
                   ori_x=None, const_alpha1=None, const_alpha2=None, const_v=None,
                   shared_expert_x=None, active_mask=None, residual=None, gamma=None,
                   eps: float = 1e-6, y=None, x_out=None, rstd=None, stream=None):
    """Combine with special experts, a shared expert and an active mask
    (bool [T] or [T, k]); with ``residual`` also Add + RMSNorm. Returns ``y``,
    or ``(y, x_out, rstd)`` with a residual."""
    T, k = weights.shape
    H = out_disp.shape[1]
    dev = out_disp.device
    y = y if y is not None else torch.empty((T, H), dtype=dtype, device=dev)
    mask = None if active_mask is None else active_mask.to(torch.uint8).contiguous()
    ex = CombineExtras(_ptr(expert_indices), int(num_experts), int(zero_experts),
                       int(copy_experts), int(const_experts), _ptr(ori_x), _ptr(const_alpha1),
                       _ptr(const_alpha2), _ptr(const_v), _ptr(shared_expert_x), _ptr(mask),
                       0 if mask is None else mask.dim())
    if residual is not None:
        x_out = x_out if x_out is not None else torch.empty((T, H), dtype=dtype, device=dev)
        rstd = rstd if rstd is not None else torch.empty(T, dtype=torch.float32, device=dev)
    rc = load_library().moe_combine_v2(
        _ptr(out_disp), _code(out_disp.dtype), _ptr(weights), _code(weights.dtype),
        _ptr(row_of), ctypes.byref(ex), _ptr(residual), _ptr(gamma),
        _code(gamma.dtype) if gamma is not None else 0, float(eps), T, k, H, _ptr(y),
        _code(dtype), _ptr(x_out), _ptr(rstd), _stream(stream))
    _check(rc, "moe_combine_v2")
    return y if residual is None else (y, x_out, rstd)


def moe_rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float, y=None, rstd=None,
                stream=None):
    """RMSNorm over the last axis of ``x [rows, H]``; returns ``(y, rstd)``."""
    rows, H = x.shape
    y = y if y is not None else torch.empty_like(x)
    rstd = rstd if rstd is not None else torch.empty(rows, dtype=torch.float32, device=x.device)
    rc = load_library().moe_rmsnorm(_ptr(x), _code(x.dtype), _ptr(gamma), _code(gamma.dtype),
                                    float(eps), rows, H, _ptr(y), _ptr(rstd), _stream(stream))
    _check(rc, "moe_rmsnorm")
    return y, rstd


def moe_forward_workspace_size(T: int, H: int, I: int, E: int, top_k: int,
                               dtype: torch.dtype, logits_dtype: torch.dtype,
                               deterministic: bool = False) -> int:
    flags = MOE_FORWARD_DETERMINISTIC if deterministic else 0
    return int(load_library().moe_forward_workspace_size_ex(
        T, H, I, E, top_k, _code(dtype), _code(logits_dtype), flags))


def moe_forward_workspace_layout(T: int, H: int, I: int, E: int, top_k: int,
                                 dtype: torch.dtype, logits_dtype: torch.dtype,
                                 deterministic: bool = False) -> dict:
    """Byte offsets of the routing plan and dispatch map inside the one-call
    forward's workspace (``moe_forward_layout``)."""
    lay = ForwardLayout()
    flags = MOE_FORWARD_DETERMINISTIC if deterministic else 0
    rc = load_library().moe_forward_workspace_layout(T, H, I, E, top_k, _code(dtype),
                                                     _code(logits_dtype), flags,
                                                     ctypes.byref(lay))
    _check(rc, "moe_forward_workspace_layout")
    return {n: int(getattr(lay, n)) for n, _ in ForwardLayout._fields_}


def _event_handle(ev) -> ctypes.c_void_p:
    return ctypes.c_void_p(None) if ev is None else ctypes.c_void_p(ev.cuda_event)


def moe_forward_ex(x: torch.Tensor, logits: torch.Tensor, gate: torch.Tensor, up: torch.Tensor,
                   down: torch.Tensor, top_k: int, renormalize: bool, deterministic: bool = False,
                   sigmoid_grouped: dict | None = None, experts_begin_event=None,
                   experts_end_event=None, y=None, workspace=None,
                   stream=None) -> torch.Tensor:
    """The whole local forward with ``moe_forward_options``: a deterministic
    combine, group-limited sigmoid routing (``sigmoid_grouped``: bias, groups,
    selected_groups, group_top_two, scale) and torch.cuda.Event objects (created
    with enable_timing) recorded around the expert GEMMs."""
    T, H = x.shape
    E, I, _ = gate.shape
    dev = x.device
    y = y if y is not None else torch.empty((T, H), dtype=x.dtype, device=dev)
    ws = _workspace(moe_forward_workspace_size(T, H, I, E, top_k, x.dtype, logits.dtype,
                                               deterministic), dev, workspace)
    opt = ForwardOptions()
    opt.flags = MOE_FORWARD_DETERMINISTIC if deterministic else 0
    sg = None
    if sigmoid_grouped is not None:
        bias = sigmoid_grouped.get("bias")
        if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (E,)):
            raise ValueError("bias must be float32 of shape [E]")
        sg = SigmoidGroupedRouting(None if bias is None else _ptr(bias).value,
                                   int(sigmoid_grouped["groups"]),
                                   int(sigmoid_grouped["selected_groups"]),
                                   int(bool(sigmoid_grouped["group_top_two"])),
                                   float(sigmoid_grouped.get("scale", 1.0)))
        opt.sigmoid_grouped = ctypes.pointer(sg)
    # torch creates an event's handle on its first record and only then lets
    # elapsed_time() read it: record both here first; the library records
    # them again, later on the same stream, around the expert GEMMs
    if experts_begin_event is not None or experts_end_event is not None:
        ts = (torch.cuda.current_stream(dev) if stream is None else
              stream if isinstance(stream, torch.cuda.Stream) else
              torch.cuda.ExternalStream(int(stream)))
        for ev in (experts_begin_event, experts_end_event):
            if ev is not None:
                ev.record(ts)
    opt.experts_begin_event = _event_handle(experts_begin_event)
    opt.experts_end_event = _event_handle(experts_end_event)
    rc = load_library().moe_forward_ex(
        _ptr(x), _code(x.dtype), _ptr(logits), _code(logits.dtype), _ptr(gate),
        _ptr(up), _ptr(down), T, H, I, E, int(top_k), int(bool(renormalize)),
        _ptr(y), _ptr(ws), _nbytes(ws), ctypes.byref(opt), _stream(stream))
    _check(rc, "moe_forward_ex")
    return y


def moe_forward(x: torch.Tensor, logits: torch.Tensor, gate: torch.Tensor,
                up: torch.Tensor, down: torch.Tensor, top_k: int,
                renormalize: bool, y=None, workspace=None,
                stream=None) -> torch.Tensor:
    """The whole local forward (route, dispatch, experts, combine)."""
    T, H = x.shape
    E, I, _ = gate.shape
    dev = x.device
    y = y if y is not None else torch.empty((T, H), dtype=x.dtype, device=dev)
    ws = _workspace(moe_forward_workspace_size(T, H, I, E, top_k, x.dtype, logits.dtype),
                    dev, workspace)
    rc = load_library().moe_forward(
        _ptr(x), _code(x.dtype), _ptr(logits), _code(logits.dtype), _ptr(gate),
        _ptr(up), _ptr(down), T, H, I, E, int(top_k), int(bool(renormalize)),
        _ptr(y), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "moe_forward")
    return y


def moe_forward_sigmoid_grouped(x: torch.Tensor, logits: torch.Tensor, bias: torch.Tensor | None,
                                gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor,
                                top_k: int, groups: int, selected_groups: int,
                                group_top_two: bool, renormalize: bool, scale: float = 1.0,
                                y=None, workspace=None, stream=None) -> torch.Tensor:
    """The whole local forward with group-limited sigmoid routing."""
    T, H = x.shape
    E, I, _ = gate.shape
    dev = x.device
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (E,)):
        raise ValueError("bias must be float32 of shape [E]")
    y = y if y is not None else torch.empty((T, H), dtype=x.dtype, device=dev)
    ws = _workspace(moe_forward_workspace_size(T, H, I, E, top_k, x.dtype, logits.dtype),
                    dev, workspace)
    rc = load_library().moe_forward_sigmoid_grouped(
        _ptr(x), _code(x.dtype), _ptr(logits), _code(logits.dtype),
        None if bias is None else _ptr(bias), _ptr(gate), _ptr(up), _ptr(down), T, H, I, E,
        int(top_k), int(groups), int(selected_groups), int(bool(group_top_two)),
        int(bool(renormalize)), float(scale), _ptr(y), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "moe_forward_sigmoid_grouped")
    return y


def moe_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of every bounded device wait (0: the default 2 s)."""
    _check(load_library().moe_set_wait_limit_ns(int(limit_ns)), "moe_set_wait_limit_ns")


def moe_wait_limit_ns() -> int:
    return int(load_library().moe_wait_limit_ns())


def moe_selftest_wait_expiry(E: int, rows_per_expert: int, H: int, I: int,
                             y_acc: torch.Tensor, workspace=None, stream=None) -> None:
    """Run the bounded waits' failure path (see include/moe.h)."""
    lib = load_library()
    ws = _workspace(int(lib.moe_selftest_wait_expiry_workspace_size(E, rows_per_expert, H, I)),
                    y_acc.device, workspace)
    rc = lib.moe_selftest_wait_expiry(E, rows_per_expert, H, I, _ptr(y_acc), _ptr(ws),
                                      _nbytes(ws), _stream(stream))
    _check(rc, "moe_selftest_wait_expiry")


def moe_device_status(stream=None, clear: bool = True) -> int:
    """Synchronise ``stream`` and return the device status code (0 = OK)."""
    return int(load_library().moe_device_status(_stream(stream), int(bool(clear))))


# ---- first-order training (ruDNN user guide, section 12) -------------------

def _index_code(indices: torch.Tensor) -> int:
    if indices.dtype not in INDEX_CODES:
        raise TypeError("expert ids must be int32, int64 or uint32")
    return INDEX_CODES[indices.dtype]


def moe_router_weights(logits: torch.Tensor, indices: torch.Tensor, scoring: str = "softmax",
                       renormalize: bool = False, scale: float = 1.0, weights=None,
                       stream=None) -> torch.Tensor:
    """FP32 weights ``[T, k]`` of the fixed selection ``indices``
    (selected_router_weights)."""
    T, E = logits.shape
    k = indices.shape[1]
    weights = weights if weights is not None else torch.empty(
        (T, k), dtype=torch.float32, device=logits.device)
    rc = load_library().moe_router_weights(
        _ptr(logits), _code(logits.dtype), T, E, _ptr(indices), _index_code(indices), k,
        SCORING_CODES[scoring], int(bool(renormalize)), float(scale), _ptr(weights),
        _stream(stream))
    _check(rc, "moe_router_weights")
    return weights


def moe_router_backward(logits: torch.Tensor, indices: torch.Tensor, grad_weights: torch.Tensor,
                        scoring: str = "softmax", renormalize: bool = False, scale: float = 1.0,
                        grad_logits=None, stream=None) -> torch.Tensor:
    """Logits gradient ``[T, E]`` (logits dtype) of :func:`moe_router_weights`
    for the FP32 upstream gradient ``grad_weights [T, k]``."""
    T, E = logits.shape
    k = indices.shape[1]
    grad_logits = grad_logits if grad_logits is not None else torch.empty_like(logits)
    rc = load_library().moe_router_backward(
        _ptr(logits), _code(logits.dtype), T, E, _ptr(indices), _index_code(indices), k,
        _ptr(grad_weights), SCORING_CODES[scoring], int(bool(renormalize)), float(scale),
        _ptr(grad_logits), _stream(stream))
    _check(rc, "moe_router_backward")
    return grad_logits


def moe_combine_backward(out_disp: torch.Tensor, weights: torch.Tensor, row_of: torch.Tensor,
                         grad_y: torch.Tensor, grad_out_disp=None, grad_weights=None,
                         stream=None):
    """Backward of :func:`moe_combine`. Returns ``(grad_out_disp [T*k, H] in
    grad_y.dtype, grad_weights [T, k] FP32)``."""
    T, k = weights.shape
    H = grad_y.shape[1]
    dev = grad_y.device
    grad_out_disp = grad_out_disp if grad_out_disp is not None else torch.empty(
        (out_disp.shape[0], H), dtype=grad_y.dtype, device=dev)
    grad_weights = grad_weights if grad_weights is not None else torch.empty(
        (T, k), dtype=torch.float32, device=dev)
    rc = load_library().moe_combine_backward(
        _ptr(out_disp), _code(out_disp.dtype), _ptr(weights), _code(weights.dtype),
        _ptr(row_of), _ptr(grad_y), T, k, H, _code(grad_y.dtype), _ptr(grad_out_disp),
        _ptr(grad_weights), _stream(stream))
    _check(rc, "moe_combine_backward")
    return grad_out_disp, grad_weights


def moe_dispatch_backward(grad_x_disp: torch.Tensor, row_of: torch.Tensor, T: int, top_k: int,
                          grad_x=None, stream=None) -> torch.Tensor:
    """Sum every token's dispatched gradient rows back to ``grad_x [T, H]``."""
    H = grad_x_disp.shape[1]
    grad_x = grad_x if grad_x is not None else torch.empty(
        (T, H), dtype=grad_x_disp.dtype, device=grad_x_disp.device)
    rc = load_library().moe_dispatch_backward(
        _ptr(grad_x_disp), _code(grad_x_disp.dtype), _ptr(row_of), T, int(top_k), H,
        _ptr(grad_x), _stream(stream))
    _check(rc, "moe_dispatch_backward")
    return grad_x


def moe_experts_training_cache_size(rows: int, I: int, dtype: torch.dtype) -> int:
    return int(load_library().moe_experts_training_cache_size(rows, I, _code(dtype)))


def moe_experts_forward_training(x_disp: torch.Tensor, offsets: torch.Tensor,
                                 gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor,
                                 out_dtype: torch.dtype | None = None, out_disp=None,
                                 cache=None, stream=None):
    """SwiGLU experts that keep the backward's cache. Returns ``(out_disp,
    cache)``; ``cache`` (uint8) holds h, g, u as three ``[rows, I]`` planes."""
    rows, H = x_disp.shape
    E, I, _ = gate.shape
    dev = x_disp.device
    if out_disp is not None:
        out_dtype = out_disp.dtype
    out_dtype = out_dtype or x_disp.dtype
    if out_disp is None:
        out_disp = torch.empty((rows, H), dtype=out_dtype, device=dev)
    cache = _workspace(moe_experts_training_cache_size(rows, I, x_disp.dtype), dev, cache)
    rc = load_library().moe_experts_forward_training(
        _ptr(x_disp), _ptr(offsets), rows, _ptr(gate), _ptr(up), _ptr(down), E, H, I,
        _code(x_disp.dtype), _ptr(out_disp), _code(out_dtype), _ptr(cache), _nbytes(cache),
        _stream(stream))
    _check(rc, "moe_experts_forward_training")
    return out_disp, cache


def moe_experts_backward_workspace_size(rows: int, E: int, H: int, I: int,
                                        dtype: torch.dtype) -> int:
    return int(load_library().moe_experts_backward_workspace_size(rows, E, H, I, _code(dtype)))


def moe_experts_backward(x_disp: torch.Tensor, offsets: torch.Tensor, gate: torch.Tensor,
                         up: torch.Tensor, down: torch.Tensor, cache: torch.Tensor,
                         grad_out: torch.Tensor, grad_x_disp=None, grad_gate=None,
                         grad_up=None, grad_down=None, workspace=None, stream=None):
    """Backward of the SwiGLU experts. Returns ``(grad_x_disp [rows, H],
    grad_gate [E, I, H], grad_up [E, I, H], grad_down [E, H, I])``, the
    weight gradients in FP32."""
    rows, H = x_disp.shape
    E, I, _ = gate.shape
    dev = x_disp.device
    f32 = torch.float32
    grad_x_disp = grad_x_disp if grad_x_disp is not None else torch.empty_like(x_disp)
    grad_gate = grad_gate if grad_gate is not None else torch.empty((E, I, H), dtype=f32, device=dev)
    grad_up = grad_up if grad_up is not None else torch.empty((E, I, H), dtype=f32, device=dev)
    grad_down = grad_down if grad_down is not None else torch.empty((E, H, I), dtype=f32, device=dev)
    ws = _workspace(moe_experts_backward_workspace_size(rows, E, H, I, x_disp.dtype), dev,
                    workspace)
    rc = load_library().moe_experts_backward(
        _ptr(x_disp), _ptr(offsets), rows, _ptr(gate), _ptr(up), _ptr(down), E, H, I,
        _code(x_disp.dtype), _ptr(cache), _ptr(grad_out), _ptr(grad_x_disp), _ptr(grad_gate),
        _ptr(grad_up), _ptr(grad_down), _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "moe_experts_backward")
    return grad_x_disp, grad_gate, grad_up, grad_down
