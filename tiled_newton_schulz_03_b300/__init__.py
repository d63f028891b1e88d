"""HiMuon tiled Newton-Schulz for B300: Python binding of ``libhimuon.so``.

The library (C ABI, ``include/himuon.h``) does all the work in its own CUDA
kernels; this module only marshals torch tensors (device pointers, shapes,
strides, dtypes) and the current CUDA stream into the C calls. There is no
fallback: if the library is missing or the device is not an sm_103 GPU, the
calls raise.

Method: "Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
Optimization" (abstract): each momentum-gradient matrix is cut into T x T tiles,
the same K-step Newton-Schulz map runs on every tile independently, and the
results are reassembled; tiles of many layers are batched into one launch,
launches are bounded in memory, and T may change between optimizer steps.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "QUINTIC", "HimuonError", "Handle", "library_path", "load_library", "tiled_ns",
    "tiled_ns_batched", "step", "ns_flops", "schedule_tile", "TSchedule",
    "device_error", "set_wait_limit", "wait_selftest", "EXPORTED_SYMBOLS", "default_handle",
    "tiled_ns_fp32_noalloc", "NOALLOC_SCRATCH_BYTES",
]

QUINTIC = (3.4445, -4.7750, 2.0315)

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libhimuon.so"

# Every symbol include/himuon.h declares.
EXPORTED_SYMBOLS = [
    "himuon_create", "himuon_destroy", "himuon_default_ns_params", "himuon_tiled_ns",
    "himuon_tiled_ns_batched", "himuon_step", "himuon_schedule_tile", "himuon_ns_flops",
    "himuon_device_error", "himuon_set_wait_limit", "himuon_wait_selftest",
    "himuon_last_error_string", "himuon_version", "himuon_launch_count",
    "himuon_tiled_ns_fp32_noalloc",
]

# Size of the fixed device scratch of himuon_tiled_ns_fp32_noalloc (HIMUON_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 16 << 20

_STATUS = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "TIMEOUT",
           5: "NO_DEVICE", 6: "OUT_OF_MEMORY"}
_DTYPE = {torch.bfloat16: 0, torch.float32: 1}
_NORM = {"tile": 0, "matrix": 1, "none": 2}
_PATH = {"auto": 0, "tensor": 1, "fp32": 2}
_SCALE = {"sqrt_aspect": 0, "none": 1}


class HimuonError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = _STATUS.get(status, str(status))
        super().__init__(f"himuon: {self.status_name}: {message}")


class NSParams(ctypes.Structure):
    _fields_ = [("a", ctypes.c_float), ("b", ctypes.c_float), ("c", ctypes.c_float),
                ("norm", ctypes.c_int32), ("eps", ctypes.c_float), ("path", ctypes.c_int32),
                ("step_coeffs", ctypes.POINTER(ctypes.c_float))]


class Matrix(ctypes.Structure):
    _fields_ = [("g", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("H", ctypes.c_int64), ("W", ctypes.c_int64),
                ("ldg", ctypes.c_int64), ("ldo", ctypes.c_int64),
                ("gtype", ctypes.c_int32), ("otype", ctypes.c_int32)]


class Param(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("g", ctypes.c_void_p), ("m", ctypes.c_void_p),
                ("H", ctypes.c_int64), ("W", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("ldg", ctypes.c_int64), ("ldm", ctypes.c_int64),
                ("wtype", ctypes.c_int32), ("gtype", ctypes.c_int32), ("mtype", ctypes.c_int32)]


class StepParams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("mu", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("nesterov", ctypes.c_int32), ("scale_mode", ctypes.c_int32)]


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def load_library():
    """Loads libhimuon.so (built in-tree) and declares its signatures."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise HimuonError(5, f"{path} is not built; run `python -m tiled_newton_schulz_03_b300.build`")
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "himuon_create": (I32, [ctypes.POINTER(ctypes.c_void_p)]),
            "himuon_destroy": (I32, [P]),
            "himuon_default_ns_params": (None, [ctypes.POINTER(NSParams)]),
            "himuon_tiled_ns": (I32, [P, P, I64, I64, I64, I32, I32, I32,
                                      ctypes.POINTER(NSParams), P, I64, I32, P]),
            "himuon_tiled_ns_batched": (I32, [P, ctypes.POINTER(Matrix), I32, I32, I32,
                                              ctypes.POINTER(NSParams), SZ, P]),
            "himuon_step": (I32, [P, ctypes.POINTER(Param), I32, I32, I32, ctypes.POINTER(NSParams),
                                  ctypes.POINTER(StepParams), SZ, P]),
            "himuon_schedule_tile": (I32, [ctypes.POINTER(I64), ctypes.POINTER(I32), I32, I64]),
            "himuon_ns_flops": (ctypes.c_double, [I64, I64, I32, I32]),
            "himuon_device_error": (I32, [P, P, ctypes.POINTER(I32)]),
            "himuon_set_wait_limit": (I32, [P, ctypes.c_uint64]),
            "himuon_wait_selftest": (I32, [P, P]),
            "himuon_last_error_string": (ctypes.c_char_p, []),
            "himuon_version": (I32, []),
            "himuon_launch_count": (I64, [P]),
            "himuon_tiled_ns_fp32_noalloc": (I32, [P, I64, I64, I64, I32, I32, I32,
                                                   ctypes.POINTER(NSParams), P, I64, I32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        msg = load_library().himuon_last_error_string().decode(errors="replace")
        raise HimuonError(status, msg)


class Handle:
    """A libhimuon handle (device workspace) bound to one CUDA device."""

    def __init__(self, device=None):
        lib = load_library()
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.device = dev
        self._ptr = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _check(lib.himuon_create(ctypes.byref(self._ptr)))

    @property
    def ptr(self):
        return self._ptr

    def launch_count(self) -> int:
        """Kernels launched through this handle so far."""
        return int(load_library().himuon_launch_count(self._ptr))

    def close(self):
        if self._ptr:
            with torch.cuda.device(self.device):
                load_library().himuon_destroy(self._ptr)
            self._ptr = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_handles: dict[int, Handle] = {}


def _default_handle(device: torch.device) -> Handle:
    idx = device.index if device.index is not None else torch.cuda.current_device()
    h = _handles.get(idx)
    if h is None:
        h = _handles[idx] = Handle(torch.device("cuda", idx))
    return h


def _stream_ptr(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _mat_info(t: torch.Tensor, name: str):
    """(pointer, H, W, leading dimension, dtype code) of a row-major 2-D CUDA matrix.

    Reads the shape and the strides as one tuple each: a step over hundreds of
    matrices spends its host time here."""
    try:
        shape, strides, dt = t.shape, t.stride(), _DTYPE.get(t.dtype)
        cuda = t.is_cuda
    except AttributeError:
        raise HimuonError(1, f"{name} must be a CUDA tensor") from None
    if not cuda:
        raise HimuonError(1, f"{name} must be a CUDA tensor")
    if len(shape) != 2:
        raise HimuonError(1, f"{name} must be 2-D")
    if dt is None:
        raise HimuonError(1, f"{name} must be bfloat16 or float32")
    H, W = shape
    if W > 1 and strides[1] != 1:
        raise HimuonError(1, f"{name} must be row-major (stride(1) == 1)")
    return t.data_ptr(), H, W, (strides[0] if H > 1 else max(W, 1)), dt


def _step_schedule(coeffs, K: int):
    """None for one (a, b, c) triple used at every step; else the flat list of
    K per-step triples (a_k, b_k, c_k)."""
    items = list(coeffs)
    if len(items) == 3 and all(not isinstance(v, (list, tuple)) for v in items):
        return None
    if len(items) != K or any(len(t) != 3 for t in items):
        raise HimuonError(1, f"coeffs: one (a, b, c) triple, or exactly K = {K} triples")
    return [float(v) for t in items for v in t]


def _ns_params(coeffs, norm, eps, path, K: int) -> NSParams:
    """ctypes parameters of the NS map. ``coeffs`` is one (a, b, c) triple for
    every step, or a list of K triples (a per-step schedule)."""
    if norm not in _NORM:
        raise HimuonError(1, f"unknown norm mode {norm!r}")
    if path not in _PATH:
        raise HimuonError(1, f"unknown path {path!r}")
    sched = _step_schedule(coeffs, int(K))
    if sched is None:
        a, b, c = (float(v) for v in coeffs)
        return NSParams(a, b, c, _NORM[norm], float(eps), _PATH[path], None)
    arr = (ctypes.c_float * len(sched))(*sched)
    p = NSParams(sched[0], sched[1], sched[2], _NORM[norm], float(eps), _PATH[path],
                 ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)))
    p._keep = arr                      # the array lives as long as the parameters
    return p


def tiled_ns(G: torch.Tensor, T: int, K: int = 5, coeffs=QUINTIC, norm: str = "tile",
             eps: float = 1e-7, out: torch.Tensor | None = None, out_dtype=None,
             path: str = "auto", handle: Handle | None = None, stream=None) -> torch.Tensor:
    """HiMuon tiled NS map of one matrix; returns ``out`` (new if not given)."""
    if out is None:
        out = torch.empty(G.shape, dtype=out_dtype or G.dtype, device=G.device)
    g, H, W, ldg, gt = _mat_info(G, "G")
    o, H2, W2, ldo, ot = _mat_info(out, "out")
    if (H2, W2) != (H, W):
        raise HimuonError(1, "out must have the shape of G")
    h = handle or _default_handle(G.device)
    p = _ns_params(coeffs, norm, eps, path, K)
    with torch.cuda.device(G.device):
        _check(load_library().himuon_tiled_ns(h.ptr, g, H, W, ldg, gt, int(T), int(K),
                                              ctypes.byref(p), o, ldo, ot,
                                              _stream_ptr(stream, G.device)))
    return out


def tiled_ns_fp32_noalloc(G: torch.Tensor, T: int, K: int = 5, coeffs=QUINTIC,
                          norm: str = "tile", eps: float = 1e-7, out: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """fp32 tiled NS of one matrix through the allocation-free entry point.

    For callers that cannot let the library allocate device memory: no handle
    is used and the library's scratch is its fixed device array. ``out`` must
    be given (this wrapper does not allocate one either); it is returned.
    Calls that overlap on the GPU share that array and must be serialised.
    """
    if out is None:
        raise HimuonError(1, "out must be given (this call allocates nothing)")
    g, H, W, ldg, gt = _mat_info(G, "G")
    o, H2, W2, ldo, ot = _mat_info(out, "out")
    if (H2, W2) != (H, W):
        raise HimuonError(1, "out must have the shape of G")
    p = _ns_params(coeffs, norm, eps, "fp32", K)
    with torch.cuda.device(G.device):
        _check(load_library().himuon_tiled_ns_fp32_noalloc(g, H, W, ldg, gt, int(T), int(K),
                                                           ctypes.byref(p), o, ldo, ot,
                                                           _stream_ptr(stream, G.device)))
    return out


def tiled_ns_batched(Gs, T: int, K: int = 5, coeffs=QUINTIC, norm: str = "tile",
                     eps: float = 1e-7, outs=None, out_dtype=None, path: str = "auto",
                     chunk_bytes: int = 0, handle: Handle | None = None, stream=None):
    """Cross-layer batch: one work list over all tiles of all matrices."""
    Gs = list(Gs)
    if not Gs:
        raise HimuonError(1, "need at least one matrix")
    if outs is None:
        outs = [torch.empty(g.shape, dtype=out_dtype or g.dtype, device=g.device) for g in Gs]
    outs = list(outs)
    if len(outs) != len(Gs):
        raise HimuonError(1, "outs and Gs differ in length")
    rows = []
    dev0 = Gs[0].device
    for i, (G, O) in enumerate(zip(Gs, outs)):
        g, H, W, ldg, gt = _mat_info(G, "Gs[%d]" % i)
        o, H2, W2, ldo, ot = _mat_info(O, "outs[%d]" % i)
        if H2 != H or W2 != W:
            raise HimuonError(1, f"outs[{i}] must have the shape of Gs[{i}]")
        if G.device != dev0 or O.device != dev0:
            raise HimuonError(1, "all matrices must be on one device")
        rows.append((g, o, H, W, ldg, ldo, gt, ot))
    arr = (Matrix * len(rows))(*rows)
    h = handle or _default_handle(Gs[0].device)
    p = _ns_params(coeffs, norm, eps, path, K)
    with torch.cuda.device(Gs[0].device):
        _check(load_library().himuon_tiled_ns_batched(h.ptr, arr, len(Gs), int(T), int(K),
                                                      ctypes.byref(p), int(chunk_bytes),
                                                      _stream_ptr(stream, Gs[0].device)))
    return outs


def step(Ws, Gs, Ms, T: int, K: int = 5, lr: float = 0.02, mu: float = 0.95,
         nesterov: bool = True, weight_decay: float = 0.0, scale_mode: str = "sqrt_aspect",
         coeffs=QUINTIC, norm: str = "tile", eps: float = 1e-7, path: str = "auto",
         chunk_bytes: int = 0, handle: Handle | None = None, stream=None):
    """One fused HiMuon optimizer step; W and M are updated in place."""
    Ws, Gs, Ms = list(Ws), list(Gs), list(Ms)
    if not (len(Ws) == len(Gs) == len(Ms)) or not Ws:
        raise HimuonError(1, "Ws, Gs and Ms must be non-empty lists of equal length")
    if scale_mode not in _SCALE:
        raise HimuonError(1, f"unknown scale mode {scale_mode!r}")
    rows = []
    for i, (Wt, G, M) in enumerate(zip(Ws, Gs, Ms)):
        w, H, W, ldw, wt = _mat_info(Wt, "Ws[%d]" % i)
        g, H2, W2, ldg, gt = _mat_info(G, "Gs[%d]" % i)
        m, H3, W3, ldm, mt = _mat_info(M, "Ms[%d]" % i)
        if not (H == H2 == H3 and W == W2 == W3):
            raise HimuonError(1, f"shapes of Ws[{i}], Gs[{i}], Ms[{i}] differ")
        rows.append((w, g, m, H, W, ldw, ldg, ldm, wt, gt, mt))
    arr = (Param * len(rows))(*rows)
    h = handle or _default_handle(Ws[0].device)
    p = _ns_params(coeffs, norm, eps, path, K)
    sp = StepParams(float(lr), float(mu), float(weight_decay), 1 if nesterov else 0, _SCALE[scale_mode])
    with torch.cuda.device(Ws[0].device):
        _check(load_library().himuon_step(h.ptr, arr, len(Ws), int(T), int(K), ctypes.byref(p),
                                          ctypes.byref(sp), int(chunk_bytes),
                                          _stream_ptr(stream, Ws[0].device)))
    return Ws, Ms


def ns_flops(H: int, W: int, T: int, K: int) -> float:
    """Algorithmic flops 6 H W T K of the tiled map."""
    return float(load_library().himuon_ns_flops(int(H), int(W), int(T), int(K)))


def schedule_tile(schedule, step_index: int) -> int:
    """T at ``step_index`` for a schedule [(start_step, T), ...]."""
    pts = list(schedule)
    n = len(pts)
    starts = (ctypes.c_int64 * max(n, 1))(*[int(s) for s, _ in pts])
    tiles = (ctypes.c_int32 * max(n, 1))(*[int(t) for _, t in pts])
    T = load_library().himuon_schedule_tile(starts, tiles, n, int(step_index))
    if T == 0:
        raise HimuonError(1, "schedule must be non-empty with increasing start steps")
    return T


class TSchedule:
    """Runtime tile-size schedule: ``TSchedule([(0, 64), (1, 128), (2, 256)])(step)``."""

    def __init__(self, points):
        self.points = [(int(s), int(t)) for s, t in points]
        schedule_tile(self.points, 0)  # validates

    def __call__(self, step_index: int) -> int:
        return schedule_tile(self.points, step_index)


def default_handle(device=None) -> Handle:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return _default_handle(dev)


def device_error(handle: Handle | None = None, stream=None, device=None) -> int:
    """Reads and clears the device error word (synchronises the stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    h = handle or _default_handle(dev)
    code = ctypes.c_int32(0)
    with torch.cuda.device(h.device):
        _check(load_library().himuon_device_error(h.ptr, _stream_ptr(stream, h.device), ctypes.byref(code)))
    return code.value


def set_wait_limit(ns: int, handle: Handle | None = None):
    h = handle or _default_handle(torch.device("cuda", torch.cuda.current_device()))
    _check(load_library().himuon_set_wait_limit(h.ptr, int(ns)))


def wait_selftest(handle: Handle | None = None, stream=None):
    h = handle or _default_handle(torch.device("cuda", torch.cuda.current_device()))
    with torch.cuda.device(h.device):
        _check(load_library().himuon_wait_selftest(h.ptr, _stream_ptr(stream, h.device)))
