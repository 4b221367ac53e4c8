"""Python binding of librrs, the GB300 row-wise softmax and row-sum library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/rrs.h``.  There is no CPU or
PyTorch fallback -- if the library is not built, every call raises.

Two layers, with the C ABI's names:

* ``softmax_rows(x, y=None)``, ``log_softmax_rows``, ``row_sum(x, out=None)``,
  ``row_max``, ``row_mean`` take CUDA fp32 tensors (2-D, unit column stride;
  x and y may have different row strides, and y may be x itself) and enqueue
  on the current torch stream.
* ``softmax_rows_ptr``, ``softmax_rows_ex_ptr``, ``row_sum_ptr``, ... take raw
  device addresses, sizes and a ``cudaStream_t`` handle, exactly like the C
  functions.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB_PATH

__all__ = [
    "RRSError", "load_library", "softmax_rows", "log_softmax_rows", "row_sum", "row_max",
    "row_mean", "softmax_rows_ptr", "softmax_rows_ex_ptr", "log_softmax_rows_ptr", "row_sum_ptr",
    "row_max_ptr", "row_mean_ptr", "LOG_SOFTMAX", "softmax_cols", "softmax_cols_ptr",
    "force_cols_path", "plan_softmax_cols", "COLS_PATHS", "gelu", "gelu_ptr", "attention",
    "attention_ptr",
    "device_error", "release_workspace", "force_path", "plan_softmax", "plan_row_sum",
    "occupancy", "waves", "PATHS", "SUM_PATHS", "STATUS", "LIB_PATH",
]

STATUS = {0: "RRS_OK", 1: "RRS_ERR_INVALID_ARG", 2: "RRS_ERR_ALIAS", 3: "RRS_ERR_CUDA",
          4: "RRS_ERR_TIMEOUT", 5: "RRS_ERR_NOMEM", 6: "RRS_ERR_UNSUPPORTED"}
LOG_SOFTMAX = 1  # flag bit of softmax_rows_ex
PATHS = {"auto": -1, "two_phase": 0, "row_regs": 1, "row_staged": 2, "cluster": 3, "grid": 4, "two_pass": 5}
SUM_PATHS = {"auto": -1, "row": 0, "split": 1}
COLS_PATHS = {"auto": -1, "two_phase": 0, "cluster": 1, "band": 2, "two_pass": 3}
PATH_NAMES = {v: k for k, v in PATHS.items()}
SUM_PATH_NAMES = {v: k for k, v in SUM_PATHS.items()}
COLS_PATH_NAMES = {v: k for k, v in COLS_PATHS.items()}


class RRSError(RuntimeError):
    """A non-OK status from librrs."""

    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


class Plan(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32), ("threads", ctypes.c_int32), ("grid", ctypes.c_int64),
        ("cluster", ctypes.c_int32), ("vec", ctypes.c_int32), ("warps_per_row", ctypes.c_int32),
        ("rows_per_cta", ctypes.c_int32), ("ctas_per_row", ctypes.c_int64),
        ("chunk", ctypes.c_int64), ("rounds", ctypes.c_int64), ("smem_bytes", ctypes.c_int32),
        ("vector_io", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("stages", ctypes.c_int32), ("tile", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_lock = threading.Lock()

_I64 = ctypes.c_int64
_P = ctypes.c_void_p

_SIGNATURES = {
    "softmax_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "softmax_rows_ex": (ctypes.c_int, [_P, _I64, _P, _I64, _I64, _I64, ctypes.c_int, _P]),
    "log_softmax_rows": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "row_max": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "gelu": (ctypes.c_int, [_P, _P, _I64, _P]),
    "attention_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, ctypes.c_int,
                                     ctypes.c_float, _P]),
    "softmax_cols": (ctypes.c_int, [_P, _I64, _P, _I64, _I64, _I64, ctypes.c_int, _P]),
    "rrs_force_cols_path": (ctypes.c_int, [ctypes.c_int]),
    "rrs_plan_softmax_cols": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.POINTER(Plan)]),
    "row_mean": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "softmax_rows_noalloc": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "row_sum": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _P]),
    "rrs_device_error": (ctypes.c_int, [_P]),
    "rrs_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "rrs_last_error": (ctypes.c_char_p, []),
    "rrs_release_workspace": (ctypes.c_int, []),
    "rrs_force_path": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "rrs_inject_fault": (ctypes.c_int, [ctypes.c_int]),
    "rrs_cols_two_pass_item": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64)]),
    "rrs_test_occupy": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _I64, _P]),
    "rrs_plan_softmax": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(Plan)]),
    "rrs_plan_row_sum": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(Plan)]),
    "rrs_occupancy": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "rrs_waves": (_I64, [_I64, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "rrs_version": (ctypes.c_int, []),
}


def load_library(path: str | None = None):
    """Load librrs.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"librrs.so is not built ({p} missing): run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        detail = load_library().rrs_last_error().decode(errors="replace")
        raise RRSError(status, where, detail)


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------ raw pointers ----

def softmax_rows_ptr(x: int, y: int, M: int, N: int, ld: int, stream: int = 0) -> None:
    """C ``softmax_rows`` on raw device addresses; raises :class:`RRSError` on failure."""
    _check(load_library().softmax_rows(x, y, M, N, ld, stream), "softmax_rows")


def softmax_rows_ex_ptr(x: int, ldx: int, y: int, ldy: int, M: int, N: int, flags: int = 0,
                        stream: int = 0) -> None:
    """C ``softmax_rows_ex``: separate row strides, in place when y == x, LOG_SOFTMAX flag."""
    _check(load_library().softmax_rows_ex(x, ldx, y, ldy, M, N, flags, stream), "softmax_rows_ex")


def softmax_cols_ptr(x: int, ldx: int, y: int, ldy: int, M: int, N: int, flags: int = 0,
                     stream: int = 0) -> None:
    """C ``softmax_cols``: softmax down each column (LOG_SOFTMAX flag for the log form)."""
    _check(load_library().softmax_cols(x, ldx, y, ldy, M, N, flags, stream), "softmax_cols")


def attention_ptr(q: int, k: int, v: int, o: int, lse: int, BH: int, L: int, S: int, d: int,
                  causal: bool = False, scale: float = 0.0, stream: int = 0) -> None:
    """C ``attention_fwd`` on raw device addresses (bf16 q, k, v; fp32 o and lse)."""
    _check(load_library().attention_fwd(q, k, v, o, lse or None, BH, L, S, d, int(bool(causal)),
                                        float(scale), stream), "attention_fwd")


def gelu_ptr(x: int, y: int, n: int, stream: int = 0) -> None:
    """C ``gelu`` on raw device addresses (n contiguous floats)."""
    _check(load_library().gelu(x, y, n, stream), "gelu")


def log_softmax_rows_ptr(x: int, y: int, M: int, N: int, ld: int, stream: int = 0) -> None:
    """C ``log_softmax_rows`` on raw device addresses."""
    _check(load_library().log_softmax_rows(x, y, M, N, ld, stream), "log_softmax_rows")


def row_sum_ptr(x: int, out: int, M: int, N: int, ld: int, stream: int = 0) -> None:
    """C ``row_sum`` on raw device addresses; raises :class:`RRSError` on failure."""
    _check(load_library().row_sum(x, out, M, N, ld, stream), "row_sum")


def row_max_ptr(x: int, out: int, M: int, N: int, ld: int, stream: int = 0) -> None:
    """C ``row_max`` on raw device addresses."""
    _check(load_library().row_max(x, out, M, N, ld, stream), "row_max")


def row_mean_ptr(x: int, out: int, M: int, N: int, ld: int, stream: int = 0) -> None:
    """C ``row_mean`` on raw device addresses."""
    _check(load_library().row_mean(x, out, M, N, ld, stream), "row_mean")


# ----------------------------------------------------------------- tensors ----

def _rows_view(t, name: str):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D (M x N)")
    M, N = t.shape
    if N > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride")
    ld = t.stride(0) if M > 1 else max(N, 1)
    return M, N, ld


def softmax_rows(x, y=None, stream=None, log=False):
    """Row-wise softmax (``log=True``: log-softmax) of a CUDA fp32 ``M x N`` tensor.

    ``y`` (allocated with x's row stride if None) must have x's shape; its row
    stride may differ, and ``y`` may be ``x`` itself (in place).  Enqueued on
    ``stream`` (default: the current torch stream); returns ``y``.
    """
    import torch
    M, N, ld = _rows_view(x, "x")
    if y is None:
        y = torch.empty_strided((M, N), (ld, 1), dtype=x.dtype, device=x.device)
    My, Ny, ldy = _rows_view(y, "y")
    if (My, Ny) != (M, N):
        raise ValueError("y must match x's shape")
    with torch.cuda.device(x.device):
        softmax_rows_ex_ptr(x.data_ptr(), ld, y.data_ptr(), ldy, M, N, LOG_SOFTMAX if log else 0,
                            _stream_handle(stream))
    return y


def softmax_cols(x, y=None, stream=None, log=False):
    """Softmax down each column of a CUDA fp32 ``M x N`` tensor (``log=True``: log form).

    Same tensor rules as :func:`softmax_rows`; returns ``y``.
    """
    import torch
    M, N, ld = _rows_view(x, "x")
    if y is None:
        y = torch.empty_strided((M, N), (ld, 1), dtype=x.dtype, device=x.device)
    My, Ny, ldy = _rows_view(y, "y")
    if (My, Ny) != (M, N):
        raise ValueError("y must match x's shape")
    with torch.cuda.device(x.device):
        softmax_cols_ptr(x.data_ptr(), ld, y.data_ptr(), ldy, M, N, LOG_SOFTMAX if log else 0,
                         _stream_handle(stream))
    return y


def attention(q, k, v, causal=False, scale=0.0, stream=None, want_lse=True):
    """Fused attention forward of CUDA bf16 tensors q [..., L, d], k and v [..., S, d].

    Returns (O fp32 [..., L, d], LSE fp32 [..., L] or None).  scale 0 means 1/sqrt(d).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a CUDA bfloat16 tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    L, d = q.shape[-2], q.shape[-1]
    S = k.shape[-2]
    if k.shape[-1] != d or v.shape != k.shape or q.shape[:-2] != k.shape[:-2]:
        raise ValueError("q [..., L, d], k and v [..., S, d] with the same leading dims")
    BH = int(q.numel() // max(L * d, 1)) if L * d else 0
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device) if want_lse else None
    with torch.cuda.device(q.device):
        attention_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                      lse.data_ptr() if lse is not None else 0, BH, L, S, d, causal, scale,
                      _stream_handle(stream))
    return o, lse


def gelu(x, y=None, stream=None):
    """Elementwise GeLU (tanh approximation) of a contiguous CUDA fp32 tensor; ``y`` may be ``x``."""
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
        raise ValueError("x must be a CUDA float32 tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or not y.is_contiguous() or y.dtype != torch.float32 or not y.is_cuda:
        raise ValueError("y must be a contiguous CUDA float32 tensor of x's shape")
    with torch.cuda.device(x.device):
        gelu_ptr(x.data_ptr(), y.data_ptr(), x.numel(), _stream_handle(stream))
    return y


def log_softmax_rows(x, y=None, stream=None):
    """Row-wise log-softmax, log y = (x - m) - log(s); see :func:`softmax_rows`."""
    return softmax_rows(x, y, stream, log=True)


def _reduce(fn, name, x, out, stream):
    import torch
    M, N, ld = _rows_view(x, "x")
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=x.device)
    if not out.is_cuda or out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA float32 tensor of M elements")
    with torch.cuda.device(x.device):
        fn(x.data_ptr(), out.data_ptr(), M, N, ld, _stream_handle(stream))
    return out


def row_sum(x, out=None, stream=None):
    """Sum of each row of a CUDA fp32 ``M x N`` tensor into ``out`` (M floats; allocated if None)."""
    return _reduce(row_sum_ptr, "row_sum", x, out, stream)


def row_max(x, out=None, stream=None):
    """Max of each row (NaN if the row holds one; -inf for N == 0)."""
    return _reduce(row_max_ptr, "row_max", x, out, stream)


def row_mean(x, out=None, stream=None):
    """Mean of each row (NaN for N == 0)."""
    return _reduce(row_mean_ptr, "row_mean", x, out, stream)


# ------------------------------------------------------------------- misc ----

def device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error status."""
    return load_library().rrs_device_error(_stream_handle(stream))


def release_workspace() -> None:
    _check(load_library().rrs_release_workspace(), "rrs_release_workspace")


def force_path(softmax: str | int = "auto", row_sum: str | int = "auto") -> None:
    """Force an execution path for later calls ('auto' restores the planner)."""
    sp = PATHS[softmax] if isinstance(softmax, str) else int(softmax)
    rp = SUM_PATHS[row_sum] if isinstance(row_sum, str) else int(row_sum)
    _check(load_library().rrs_force_path(sp, rp), "rrs_force_path")


def plan_softmax(M, N, ld=None, vector_ok=True, sm_count=152, smem_optin=232448) -> dict:
    """The planner's decision for this shape (pure host logic, no GPU)."""
    p = Plan()
    _check(load_library().rrs_plan_softmax(M, N, N if ld is None else ld, int(vector_ok), sm_count,
                                           smem_optin, ctypes.byref(p)), "rrs_plan_softmax")
    d = p.as_dict()
    d["path_name"] = PATH_NAMES.get(d["path"], "?")
    return d


def force_cols_path(path: str | int = "auto") -> None:
    """Force a softmax_cols path for later calls ('auto' restores the planner)."""
    cp = COLS_PATHS[path] if isinstance(path, str) else int(path)
    _check(load_library().rrs_force_cols_path(cp), "rrs_force_cols_path")


def plan_softmax_cols(M, N, ld=None, vector_ok=True, sm_count=152, smem_optin=232448) -> dict:
    """The column planner's decision for this shape (pure host logic, no GPU)."""
    p = Plan()
    _check(load_library().rrs_plan_softmax_cols(M, N, N if ld is None else ld, int(vector_ok),
                                                sm_count, smem_optin, ctypes.byref(p)),
           "rrs_plan_softmax_cols")
    d = p.as_dict()
    d["path_name"] = COLS_PATH_NAMES.get(d["path"], "?")
    return d


def plan_row_sum(M, N, ld=None, vector_ok=True, sm_count=152, smem_optin=232448) -> dict:
    p = Plan()
    _check(load_library().rrs_plan_row_sum(M, N, N if ld is None else ld, int(vector_ok), sm_count,
                                           smem_optin, ctypes.byref(p)), "rrs_plan_row_sum")
    d = p.as_dict()
    d["path_name"] = SUM_PATH_NAMES.get(d["path"], "?")
    return d


def occupancy(threads: int, regs: int, sm_regs: int = 65536, max_warps: int = 64):
    """(resident blocks, resident warps, occupancy %) for a block shape."""
    b, w = ctypes.c_int(0), ctypes.c_int(0)
    bp = load_library().rrs_occupancy(threads, regs, sm_regs, max_warps, ctypes.byref(b), ctypes.byref(w))
    return b.value, w.value, bp / 100.0


def waves(blocks: int, slots: int):
    """(waves, blocks in the last wave, idle slots in it)."""
    last, idle = _I64(0), _I64(0)
    n = load_library().rrs_waves(blocks, slots, ctypes.byref(last), ctypes.byref(idle))
    return n, last.value, idle.value
