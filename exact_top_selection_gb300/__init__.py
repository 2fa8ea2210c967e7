"""Python binding of the exact row-wise FP32 Top-K C ABI (include/exact_topk.h).

Argument marshalling only: every step of the selection runs in the CUDA
kernels of ``libexact_topk.so``.  There is no fallback: if the library is
missing or fails to load, every call raises.

Method: "Sample-Guided Exact Top-K Selection for Long-Context Sparse
Attention" (sections 4-5); API shape from the HPC-Ops pull request
"feat(topk): add sample-verified exact Top-K" (section "API")::

    counter_bytes, workspace_bytes = workspace_size(num_rows, max_kv_len, top_k)
    counters = torch.zeros(counter_bytes, dtype=torch.uint8, device="cuda")
    workspace = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    topk(logits, ke, output, num_valid_rows, top_k, counters, workspace)
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "DeviceInfo", "Plan", "PlanRequest", "ExactTopK", "ExactTopKError",
    "library", "library_path", "query_device", "make_plan", "workspace_size", "topk", "run",
    "error_string", "version", "stream_floor", "FAMILY_AUTO", "FAMILY_PERSISTENT_SAMPLED", "FAMILY_KV_SPLIT",
    "FAMILY_ROW_LOCAL_EXACT", "FAMILY_CLUSTER_SPLIT", "TRACE_FIELDS", "ROUTES", "EXPORTED_SYMBOLS",
]

FAMILY_AUTO = 0
FAMILY_PERSISTENT_SAMPLED = 1
FAMILY_KV_SPLIT = 2
FAMILY_ROW_LOCAL_EXACT = 3
FAMILY_CLUSTER_SPLIT = 4
FAMILY_NAMES = {1: "persistent_sampled", 2: "kv_split", 3: "row_local_exact", 4: "cluster_split"}

ROUTES = ("pad", "primary", "band", "exact_after_band", "exact_no_band", "direct_exact", "guess",
          "guess_exact")
TRACE_FIELDS = ("route", "tau0", "tau1", "c0", "c1", "tau_star", "e0", "q0")

EXPORTED_SYMBOLS = ("exact_topk_query_device", "exact_topk_make_plan", "exact_topk_workspace_size",
                    "exact_topk", "exact_topk_run", "exact_topk_error_string",
                    "exact_topk_version", "exact_topk_kv_split_noalloc", "exact_topk_stream_floor")


class ExactTopKError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (status {code})")


class DeviceInfo(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("persistent_ctas_per_sm", ctypes.c_int32),
                ("kvsplit_ctas_per_sm", ctypes.c_int32), ("rowlocal_ctas_per_sm", ctypes.c_int32),
                ("cluster_ctas_per_sm", ctypes.c_int32)]


class PlanRequest(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("stride", ctypes.c_int32), ("dual", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("workers", ctypes.c_int32),
                ("rho0_num", ctypes.c_int32), ("rho0_den", ctypes.c_int32),
                ("rho1_num", ctypes.c_int32), ("rho1_den", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("stride", ctypes.c_int32), ("dual", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("workers", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("top_k", ctypes.c_int32), ("q0", ctypes.c_int32),
                ("q1", ctypes.c_int32), ("rho0_num", ctypes.c_int32),
                ("rho0_den", ctypes.c_int32), ("rho1_num", ctypes.c_int32),
                ("rho1_den", ctypes.c_int32), ("cand_capacity", ctypes.c_int32),
                ("sm_count", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("num_rows", ctypes.c_int64), ("max_kv_len", ctypes.c_int64),
                ("row_pitch", ctypes.c_int64), ("counter_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64)]

    def as_dict(self):
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["family_name"] = FAMILY_NAMES.get(self.family, "?")
        return d

    def __repr__(self):
        return f"Plan({self.as_dict()})"


_lib = None


def library_path() -> str:
    return os.environ.get("EXACT_TOPK_LIBRARY") or _build.LIBRARY


def library():
    """Loads libexact_topk.so (building it in-tree first if needed; the
    EXACT_TOPK_LIBRARY environment variable names another build of the same
    library to load instead); raises if impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = os.environ.get("EXACT_TOPK_LIBRARY") or _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"exact_topk CUDA library missing: {path}")
    lib = ctypes.CDLL(path)
    c_i64, c_int, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    sz = ctypes.POINTER(ctypes.c_size_t)
    lib.exact_topk_query_device.argtypes = [c_int, ctypes.POINTER(DeviceInfo)]
    lib.exact_topk_make_plan.argtypes = [c_i64, c_i64, c_i64, c_int, ctypes.POINTER(DeviceInfo),
                                         ctypes.POINTER(PlanRequest), ctypes.POINTER(Plan)]
    lib.exact_topk_workspace_size.argtypes = [c_i64, c_i64, c_int, sz, sz]
    lib.exact_topk.argtypes = [p, c_i64, c_i64, p, p, p, c_int, p, ctypes.c_size_t, p,
                               ctypes.c_size_t, p, p]
    lib.exact_topk_run.argtypes = [ctypes.POINTER(Plan), p, p, p, p, p, ctypes.c_size_t, p,
                                   ctypes.c_size_t, p, p, p]
    lib.exact_topk_error_string.argtypes = [c_int]
    lib.exact_topk_error_string.restype = ctypes.c_char_p
    lib.exact_topk_version.argtypes = []
    lib.exact_topk_kv_split_noalloc.argtypes = [p, c_i64, c_i64, p, p, p, c_int, p]
    lib.exact_topk_kv_split_noalloc.restype = c_int
    lib.exact_topk_stream_floor.argtypes = [p, c_i64, c_i64, c_i64, p, p, c_int, p]
    lib.exact_topk_stream_floor.restype = c_int
    for name in ("exact_topk_query_device", "exact_topk_make_plan", "exact_topk_workspace_size",
                 "exact_topk", "exact_topk_run", "exact_topk_version"):
        getattr(lib, name).restype = c_int
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return library().exact_topk_error_string(int(code)).decode()


def version() -> int:
    return int(library().exact_topk_version())


def _check(code: int, where: str):
    if code != 0:
        raise ExactTopKError(code, where)


def query_device(device: int = None) -> DeviceInfo:
    if device is None:
        import torch
        device = torch.cuda.current_device()
    info = DeviceInfo()
    _check(library().exact_topk_query_device(int(device), ctypes.byref(info)),
           "exact_topk_query_device")
    return info


def make_plan(num_rows, max_kv_len, top_k, row_pitch=None, device_info=None, family=0, stride=0,
              dual=-1, splits=0, workers=0, rho0=(0, 0), rho1=(0, 0)) -> Plan:
    """Host planner (pure host logic; needs a DeviceInfo, queried when omitted)."""
    if device_info is None:
        device_info = query_device()
    req = PlanRequest(int(family), int(stride), int(dual), int(splits), int(workers),
                      int(rho0[0]), int(rho0[1]), int(rho1[0]), int(rho1[1]))
    plan = Plan()
    pitch = max_kv_len if row_pitch is None else row_pitch
    _check(library().exact_topk_make_plan(int(num_rows), int(max_kv_len), int(pitch), int(top_k),
                                          ctypes.byref(device_info), ctypes.byref(req),
                                          ctypes.byref(plan)), "exact_topk_make_plan")
    return plan


def workspace_size(num_rows, max_kv_len, top_k):
    """(counter_bytes, workspace_bytes) for the current device's default plan."""
    cb, wb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(library().exact_topk_workspace_size(int(num_rows), int(max_kv_len), int(top_k),
                                               ctypes.byref(cb), ctypes.byref(wb)),
           "exact_topk_workspace_size")
    return int(cb.value), int(wb.value)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream))


def _check_tensor(t, name, dtype, device, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def topk(logits, ke, out, num_valid_rows, top_k, counters, workspace, prev_topk=None, stream=None):
    """Enqueues one exact Top-K call (default plan) on ``stream`` (default: current)."""
    import torch
    dev = logits.device
    _check_tensor(logits, "logits", torch.float32, dev, 2)
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous [num_rows, max_kv_len]")
    M, N = logits.shape
    _check_tensor(ke, "ke", torch.int32, dev, 1)
    _check_tensor(out, "out", torch.int32, dev, 2)
    if tuple(out.shape) != (M, int(top_k)) or not out.is_contiguous() or ke.shape[0] != M:
        raise ValueError("out must be contiguous [num_rows, top_k] and ke [num_rows]")
    if num_valid_rows is not None:
        _check_tensor(num_valid_rows, "num_valid_rows", torch.int32, dev)
    if prev_topk is not None:
        _check_tensor(prev_topk, "prev_topk", torch.int32, dev, 2)
        if tuple(prev_topk.shape) != (M, int(top_k)) or not prev_topk.is_contiguous():
            raise ValueError("prev_topk must be contiguous [num_rows, top_k]")
    with torch.cuda.device(dev):
        rc = library().exact_topk(_ptr(logits), M, N, _ptr(ke), _ptr(out), _ptr(num_valid_rows),
                                  int(top_k), _ptr(counters), counters.numel(), _ptr(workspace),
                                  0 if workspace is None else workspace.numel(), _ptr(prev_topk),
                                  _stream_handle(stream, dev))
    _check(rc, "exact_topk")
    return out


def run(plan: Plan, logits, ke, out, num_valid_rows, counters, workspace, prev_topk=None,
        trace=None, stream=None):
    """Enqueues one call with an explicit plan; ``trace`` optionally receives
    [num_rows, 8] int32 per-row route records."""
    import torch
    dev = logits.device
    _check_tensor(logits, "logits", torch.float32, dev, 2)
    M = logits.shape[0]
    if M != plan.num_rows or logits.stride(1) != 1 or logits.stride(0) != plan.row_pitch:
        raise ValueError("logits layout does not match the plan")
    if logits.shape[1] != plan.max_kv_len:
        raise ValueError("logits width does not match the plan")
    _check_tensor(ke, "ke", torch.int32, dev, 1)
    _check_tensor(out, "out", torch.int32, dev, 2)
    if tuple(out.shape) != (M, plan.top_k) or not out.is_contiguous():
        raise ValueError("out must be contiguous [num_rows, top_k]")
    if trace is not None:
        _check_tensor(trace, "trace", torch.int32, dev, 2)
        if tuple(trace.shape) != (M, len(TRACE_FIELDS)) or not trace.is_contiguous():
            raise ValueError("trace must be contiguous [num_rows, 8]")
    with torch.cuda.device(dev):
        rc = library().exact_topk_run(ctypes.byref(plan), _ptr(logits), _ptr(ke), _ptr(out),
                                      _ptr(num_valid_rows), _ptr(counters), counters.numel(),
                                      _ptr(workspace),
                                      0 if workspace is None else workspace.numel(),
                                      _ptr(prev_topk), _ptr(trace), _stream_handle(stream, dev))
    _check(rc, "exact_topk_run")
    return out


def stream_floor(logits, ke, splits, out=None, stream=None):
    """Enqueues the streaming-floor kernel (reads each row's valid prefix
    once, in `splits` segments per row); returns the [rows, splits] uint32
    checksums.  A measurement utility, not a selection."""
    import torch
    dev = logits.device
    _check_tensor(logits, "logits", torch.float32, dev, 2)
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous")
    M, N = logits.shape
    _check_tensor(ke, "ke", torch.int32, dev, 1)
    if out is None:
        out = torch.empty(M, int(splits), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        rc = library().exact_topk_stream_floor(_ptr(logits), M, N, logits.stride(0), _ptr(ke),
                                               _ptr(out), int(splits), _stream_handle(stream, dev))
    _check(rc, "exact_topk_stream_floor")
    return out


class ExactTopK:
    """Owns a plan plus its counter and workspace buffers for one captured shape."""

    def __init__(self, num_rows, max_kv_len, top_k, device=None, row_pitch=None, **overrides):
        import torch
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        with torch.cuda.device(self.device):
            self.plan = make_plan(num_rows, max_kv_len, top_k, row_pitch=row_pitch,
                                  device_info=query_device(self.device.index), **overrides)
        self.counters = torch.zeros(max(16, self.plan.counter_bytes), dtype=torch.uint8,
                                    device=self.device)
        self.workspace = torch.empty(max(16, self.plan.workspace_bytes), dtype=torch.uint8,
                                     device=self.device)

    def __call__(self, logits, ke, num_valid_rows=None, out=None, prev_topk=None, trace=None,
                 stream=None):
        import torch
        if out is None:
            out = torch.empty(self.plan.num_rows, self.plan.top_k, dtype=torch.int32,
                              device=self.device)
        return run(self.plan, logits, ke, out, num_valid_rows, self.counters, self.workspace,
                   prev_topk=prev_topk, trace=trace, stream=stream)
