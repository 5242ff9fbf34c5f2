"""ctypes binding of libwgrad.so (include/wgrad.h).  Argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors may be
torch tensors (their data_ptr() is passed) or plain integer device addresses.
The library must have been built (``python -m implicit_gemm_gb300.build``);
loading raises if it is missing -- there is no other code path.

A problem spec is a dict: ndim, G, N, C, K, and per-dim lists in, filt,
stride, dil, pad_l, pad_r (ndim entries, outermost first), plus in_dtype
('bf16' | 'fp16') and out_dtype ('fp32' | 'bf16' | 'fp16').
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}
MODES = {"auto": 0, "direct": 1, "atomic": 2, "deterministic": 3}
STATUS = {0: "WG_OK", 1: "WG_ERR_INVALID_ARGUMENT", 2: "WG_ERR_NOT_SUPPORTED", 3: "WG_ERR_MISALIGNED",
          4: "WG_ERR_WORKSPACE", 5: "WG_ERR_CUDA", 6: "WG_ERR_DEVICE_TIMEOUT"}


class WgProblem(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int), ("G", ctypes.c_int), ("N", ctypes.c_int), ("C", ctypes.c_int),
                ("K", ctypes.c_int), ("in_", ctypes.c_int * 3), ("filt", ctypes.c_int * 3),
                ("out", ctypes.c_int * 3), ("stride", ctypes.c_int * 3), ("dil", ctypes.c_int * 3),
                ("pad_l", ctypes.c_int * 3), ("pad_r", ctypes.c_int * 3), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int)]


class WgOptions(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int), ("mode", ctypes.c_int), ("group_merge", ctypes.c_int),
                ("cluster", ctypes.c_int), ("kernel", ctypes.c_int)]


class WgradError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


EXPORTS = ("wg_problem_normalize", "wg_workspace_size", "wg_conv_bwd_weight", "wg_check_status",
           "wg_plan_string", "wg_status_string", "wg_last_error", "wg_conv_bwd_weight_noalloc",
           "wg_set_mark_event", "wg_conv_bwd_data", "wg_bwd_data_plan_string", "wg_bwd_data_workspace_size",
           "wg_conv_bwd_weight_host", "wg_selftest_timeout")

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load():
    """Load libwgrad.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"libwgrad.so not found at {_build.LIB}; build it with "
                                   "`python -m implicit_gemm_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(_build.LIB)
            P, O = ctypes.POINTER(WgProblem), ctypes.POINTER(WgOptions)
            lib.wg_problem_normalize.argtypes = [P]
            lib.wg_workspace_size.argtypes = [P, O, ctypes.POINTER(ctypes.c_size_t)]
            lib.wg_conv_bwd_weight.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, O,
                                               ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
            lib.wg_conv_bwd_weight_noalloc.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, O,
                                                       ctypes.c_void_p]
            lib.wg_conv_bwd_weight_host.argtypes = [P] + [ctypes.c_void_p] * 6 + [O, ctypes.c_void_p, ctypes.c_size_t,
                                                                                  ctypes.c_void_p]
            lib.wg_check_status.argtypes = [ctypes.c_void_p]
            lib.wg_selftest_timeout.argtypes = [ctypes.c_void_p]
            lib.wg_set_mark_event.argtypes = [ctypes.c_void_p]
            lib.wg_conv_bwd_data.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_size_t, ctypes.c_void_p]
            lib.wg_bwd_data_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
            lib.wg_bwd_data_plan_string.argtypes = [P, ctypes.c_char_p, ctypes.c_size_t]
            lib.wg_plan_string.argtypes = [P, O, ctypes.c_char_p, ctypes.c_size_t]
            lib.wg_status_string.argtypes = [ctypes.c_int]
            lib.wg_status_string.restype = ctypes.c_char_p
            lib.wg_last_error.restype = ctypes.c_char_p
            for name in EXPORTS:
                if name not in ("wg_status_string", "wg_last_error"):
                    getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(st: int):
    if st != 0:
        raise WgradError(st, load().wg_last_error().decode())


def make_problem(spec: dict) -> WgProblem:
    p = WgProblem()
    nd = spec["ndim"]
    p.ndim, p.G, p.N, p.C, p.K = nd, spec["G"], spec["N"], spec["C"], spec["K"]
    for key, field, default in (("in", "in_", 1), ("filt", "filt", 1), ("stride", "stride", 1),
                                ("dil", "dil", 1), ("pad_l", "pad_l", 0), ("pad_r", "pad_r", 0),
                                ("out", "out", 0)):
        vals = list(spec.get(key, [default] * max(nd, 0)))
        arr = getattr(p, field)
        for i in range(3):
            arr[i] = vals[i] if i < min(nd, len(vals)) else 0
    p.in_dtype = DTYPES[spec.get("in_dtype", "bf16")]
    p.out_dtype = DTYPES[spec.get("out_dtype", "fp32")]
    return p


KERNELS = {"auto": 0, "igemm": 1, "depthwise": 2, "igemm_taps_m": 3, "igemm_taps_mn": 4, "igemm_pair": 5}


def make_options(split_k: int = 0, mode: str = "auto", group_merge: int = 0, cluster: int = 0,
                 kernel: str = "auto") -> WgOptions:
    return WgOptions(int(split_k), MODES[mode], int(group_merge), int(cluster), KERNELS[kernel])


def _addr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def wg_problem_normalize(spec: dict) -> list:
    """Derived output lengths (ndim entries)."""
    p = make_problem(spec)
    _check(load().wg_problem_normalize(ctypes.byref(p)))
    return [p.out[i] for i in range(spec["ndim"])]


def wg_workspace_size(spec: dict, split_k: int = 0, mode: str = "auto", group_merge: int = 0, *,
                      cluster: int = 0, kernel: str = "auto") -> int:
    p, o, n = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel), ctypes.c_size_t(0)
    _check(load().wg_workspace_size(ctypes.byref(p), ctypes.byref(o), ctypes.byref(n)))
    return int(n.value)


def wg_plan_string(spec: dict, split_k: int = 0, mode: str = "auto", group_merge: int = 0, *,
                   cluster: int = 0, kernel: str = "auto") -> str:
    p, o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
    buf = ctypes.create_string_buffer(2048)
    _check(load().wg_plan_string(ctypes.byref(p), ctypes.byref(o), buf, len(buf)))
    return buf.value.decode()


def wg_conv_bwd_weight(spec: dict, x, dy, dw, split_k: int = 0, mode: str = "auto", group_merge: int = 0,
                       workspace=None, ws_bytes: int | None = None, stream=None, *, cluster: int = 0, kernel: str = "auto") -> None:
    """Launch the weight gradient on `stream` (torch stream, raw handle int, or None for
    torch's current stream when torch is loaded, else the legacy default stream)."""
    p, o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else (workspace.numel() * workspace.element_size()
                                                if hasattr(workspace, "numel") else 0)
    _check(load().wg_conv_bwd_weight(ctypes.byref(p), _addr(x), _addr(dy), _addr(dw), ctypes.byref(o),
                                     _addr(workspace), int(ws_bytes), _stream_handle(stream)))


class PreparedCall:
    """wg_conv_bwd_weight with its arguments marshalled once: calling it makes one
    ctypes call.  Keeps references to the tensors it was built from."""

    def __init__(self, spec: dict, x, dy, dw, split_k: int = 0, mode: str = "auto", group_merge: int = 0,
                 workspace=None, ws_bytes: int | None = None, *, cluster: int = 0, kernel: str = "auto"):
        self._keep = (x, dy, dw, workspace)
        self.p, self.o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
        if ws_bytes is None:
            ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self.fn = load().wg_conv_bwd_weight
        self.args = (ctypes.byref(self.p), ctypes.c_void_p(_addr(x)), ctypes.c_void_p(_addr(dy)),
                     ctypes.c_void_p(_addr(dw)), ctypes.byref(self.o), ctypes.c_void_p(_addr(workspace)),
                     ctypes.c_size_t(int(ws_bytes)))

    def __call__(self, stream_handle: int | None = None) -> None:
        st = self.fn(*self.args, stream_handle)
        if st:
            _check(st)


def wg_conv_bwd_weight_host(spec: dict, x_host, dy_host, dw_host, x_dev, dy_dev, dw_dev, split_k: int = 0,
                            mode: str = "auto", group_merge: int = 0, workspace=None, ws_bytes: int | None = None,
                            stream=None, *, cluster: int = 0, kernel: str = "auto") -> None:
    """The weight gradient from host buffers (x_host, dy_host; ideally pinned) into dw_host,
    staged through the device buffers x_dev, dy_dev, dw_dev; copies overlap the compute."""
    p, o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().wg_conv_bwd_weight_host(ctypes.byref(p), _addr(x_host), _addr(dy_host), _addr(dw_host),
                                          _addr(x_dev), _addr(dy_dev), _addr(dw_dev), ctypes.byref(o),
                                          _addr(workspace), int(ws_bytes), _stream_handle(stream)))


class PreparedHostCall:
    """wg_conv_bwd_weight_host with its arguments marshalled once (one ctypes call per use)."""

    def __init__(self, spec: dict, x_host, dy_host, dw_host, x_dev, dy_dev, dw_dev, split_k: int = 0,
                 mode: str = "auto", group_merge: int = 0, workspace=None, ws_bytes: int | None = None, *,
                 cluster: int = 0, kernel: str = "auto"):
        self._keep = (x_host, dy_host, dw_host, x_dev, dy_dev, dw_dev, workspace)
        self.p, self.o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
        if ws_bytes is None:
            ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self.fn = load().wg_conv_bwd_weight_host
        self.args = (ctypes.byref(self.p), *(ctypes.c_void_p(_addr(t)) for t in (x_host, dy_host, dw_host, x_dev,
                                                                                 dy_dev, dw_dev)),
                     ctypes.byref(self.o), ctypes.c_void_p(_addr(workspace)), ctypes.c_size_t(int(ws_bytes)))

    def __call__(self, stream_handle: int | None = None) -> None:
        st = self.fn(*self.args, stream_handle)
        if st:
            _check(st)


def wg_conv_bwd_weight_noalloc(spec: dict, x, dy, dw, split_k: int = 0, mode: str = "auto", group_merge: int = 0,
                               stream=None, *, cluster: int = 0, kernel: str = "auto") -> None:
    """wg_conv_bwd_weight for callers that cannot allocate: the split-K workspace comes
    from the library's own 16 MiB device array (see include/wgrad.h)."""
    p, o = make_problem(spec), make_options(split_k, mode, group_merge, cluster, kernel)
    _check(load().wg_conv_bwd_weight_noalloc(ctypes.byref(p), _addr(x), _addr(dy), _addr(dw), ctypes.byref(o),
                                             _stream_handle(stream)))


def wg_conv_bwd_data(spec: dict, dy, w, dx, workspace=None, ws_bytes: int | None = None, stream=None) -> None:
    """Backward-data: dX (spec's out_dtype) from dY and W (spec's in_dtype); see include/wgrad.h."""
    p = make_problem(spec)
    if ws_bytes is None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().wg_conv_bwd_data(ctypes.byref(p), _addr(dy), _addr(w), _addr(dx), _addr(workspace), int(ws_bytes),
                                   _stream_handle(stream)))


def wg_bwd_data_workspace_size(spec: dict) -> int:
    p, n = make_problem(spec), ctypes.c_size_t(0)
    _check(load().wg_bwd_data_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def wg_bwd_data_plan_string(spec: dict) -> str:
    p = make_problem(spec)
    buf = ctypes.create_string_buffer(1024)
    _check(load().wg_bwd_data_plan_string(ctypes.byref(p), buf, len(buf)))
    return buf.value.decode()


class PreparedDgradCall:
    """wg_conv_bwd_data with its arguments marshalled once."""

    def __init__(self, spec: dict, dy, w, dx, workspace=None, ws_bytes: int = 0):
        self._keep = (dy, w, dx, workspace)
        self.p = make_problem(spec)
        self.fn = load().wg_conv_bwd_data
        self.args = (ctypes.byref(self.p), ctypes.c_void_p(_addr(dy)), ctypes.c_void_p(_addr(w)),
                     ctypes.c_void_p(_addr(dx)), ctypes.c_void_p(_addr(workspace)), ctypes.c_size_t(int(ws_bytes)))

    def __call__(self, stream_handle: int | None = None) -> None:
        st = self.fn(*self.args, stream_handle)
        if st:
            _check(st)


def conv_bwd_data(spec: dict, dy, w, out=None, stream=None):
    """Convenience wrapper over wg_conv_bwd_data for torch CUDA tensors: allocates dX
    (N, *in, G, C) in spec['out_dtype'] with torch, then calls the library."""
    import torch
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[spec.get("out_dtype", "fp32")]
    if out is None:
        out = torch.empty((spec["N"], *spec["in"], spec["G"], spec["C"]), dtype=tdt, device=dy.device)
    nbytes = wg_bwd_data_workspace_size(spec)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dy.device) if nbytes else None
    wg_conv_bwd_data(spec, dy, w, out, ws, nbytes, stream)
    return out


def wg_set_mark_event(event) -> None:
    """Record `event` (a torch.cuda.Event, a raw cudaEvent_t, or None to stop) after
    the main kernel of every following call from this thread (see include/wgrad.h).
    A torch event must have been recorded once, so that it exists."""
    h = None if event is None else (event if isinstance(event, int) else int(event.cuda_event))
    _check(load().wg_set_mark_event(h))


def wg_selftest_timeout(stream=None) -> None:
    """Launch the library's bounded-wait self-test (see include/wgrad.h)."""
    _check(load().wg_selftest_timeout(_stream_handle(stream)))


def wg_check_status(stream=None) -> None:
    _check(load().wg_check_status(_stream_handle(stream)))


def wg_status_string(status: int) -> str:
    return load().wg_status_string(int(status)).decode()


def wg_last_error() -> str:
    return load().wg_last_error().decode()


def _stream_handle(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except Exception:  # pragma: no cover - torch missing
            pass
        return None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def conv_bwd_weight(spec: dict, x, dy, split_k: int = 0, mode: str = "auto", group_merge: int = 0, out=None,
                    stream=None, *, cluster: int = 0, kernel: str = "auto"):
    """Convenience wrapper over wg_conv_bwd_weight for torch CUDA tensors: allocates dW
    (G, K, *filt, C) in spec['out_dtype'] and the workspace it needs with torch, then calls
    the library."""
    import torch
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}[spec.get("out_dtype", "fp32")]
    if out is None:
        out = torch.empty((spec["G"], spec["K"], *spec["filt"], spec["C"]), dtype=tdt, device=x.device)
    nbytes = wg_workspace_size(spec, split_k, mode, group_merge, cluster=cluster, kernel=kernel)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device) if nbytes else None
    wg_conv_bwd_weight(spec, x, dy, out, split_k, mode, group_merge, ws, nbytes, stream, cluster=cluster,
                       kernel=kernel)
    return out
