"""ctypes binding of the C ABI in include/dep_projection.h (marshalling only).

Every function keeps the C name and takes the same arguments; tensors may be
passed as torch tensors (BF16, contiguous, on the plan's device) or as raw
integer addresses.  Each step of the projection runs in the library's CUDA
kernels; nothing here computes.  The library must have been built (see
``skinny_bf16_split_gb300.build``): there is no fallback, and loading fails
loudly when it is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdep_projection.so")

DEP_OK = 0
DEP_ERR_INVALID_ARG = 1
DEP_ERR_UNSUPPORTED = 2
DEP_ERR_MISALIGNED = 3
DEP_ERR_CUDA = 4
DEP_ERR_OOM = 5
DEP_ERR_TIMEOUT = 6
DEP_ERR_INTERNAL = 7
DEP_ERR_IO = 8

DEP_KIND_SPLITK_FMA = 1
DEP_KIND_TC = 2
DEP_KIND_ROWS = 3
DEP_KIND_TC_SPLIT = 4
DEP_KIND_TC_WIDE = 5
DEP_KIND_TC_CLUSTER = 6
DEP_KIND_TC_XM = 7
DEP_KIND_WARP_MMA = 8
DEP_PLAN_DEFAULT = 0
DEP_PLAN_TUNE = 1
DEP_PLAN_PDL = 2
DEP_PLAN_KEEP_PIECES = 4

DEP_DEV_TIMEOUT_PRODUCER = 1
DEP_DEV_TIMEOUT_CONSUMER = 2
DEP_DEV_TIMEOUT_MMA = 3
DEP_DEV_TIMEOUT_EPILOGUE = 4
DEP_DEV_BOUNDS = 5

# Every symbol include/dep_projection.h declares.
EXPORTS = (
    "dep_projection_plan", "dep_projection_plan_host", "dep_projection_run",
    "dep_projection_run_tactic", "dep_projection_run_host", "dep_projection_plan_query",
    "dep_projection_plan_table", "dep_projection_plan_set", "dep_projection_plan_workspace",
    "dep_projection_plan_save", "dep_projection_plan_load", "dep_projection_plan_destroy",
    "dep_projection_device_status", "dep_projection_selftest_timeout", "dep_bins_index",
    "dep_status_string", "dep_projection_version", "dep_projection_run_static",
    "dep_projection_plan_partials", "dep_projection_plan_exchange", "dep_projection_probe_read",
    "dep_projection_plan_selftest_exchange",
)


class dep_tactic_t(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in
                ("max_rows", "kind", "ctas", "tile_n", "tile_k", "stages", "cols", "splits")]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}

    def __repr__(self):
        return f"dep_tactic_t({self.as_dict()})"


class DepError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dep_status_string(status)} (status {status})")


_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with skinny_bf16_split_gb300.build.build() "
            "(there is no fallback implementation)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    P = ctypes.POINTER
    sig = {
        "dep_projection_plan": ([i64, i64, P(i32), i32, u32, P(vp)], i32),
        "dep_projection_plan_host": ([i64, i64, P(i32), i32, i32, P(vp)], i32),
        "dep_projection_run": ([vp, vp, vp, vp, i32, vp], i32),
        "dep_projection_run_tactic": ([vp, P(dep_tactic_t), vp, vp, vp, i32, vp], i32),
        "dep_projection_run_host": ([vp, vp, vp, vp, i32, vp], i32),
        "dep_projection_plan_query": ([vp, i32, P(dep_tactic_t)], i32),
        "dep_projection_plan_table": ([vp, P(dep_tactic_t), i32, P(i32)], i32),
        "dep_projection_plan_set": ([vp, P(dep_tactic_t)], i32),
        "dep_projection_plan_workspace": ([vp, P(ctypes.c_size_t)], i32),
        "dep_projection_plan_save": ([vp, ctypes.c_char_p], i32),
        "dep_projection_plan_load": ([ctypes.c_char_p, i64, i64, P(vp)], i32),
        "dep_projection_plan_destroy": ([vp], None),
        "dep_projection_device_status": ([vp, vp, P(i32)], i32),
        "dep_projection_selftest_timeout": ([i32, P(i32)], i32),
        "dep_bins_index": ([P(i32), i32, i32], i32),
        "dep_status_string": ([i32], ctypes.c_char_p),
        "dep_projection_version": ([], i32),
        "dep_projection_run_static": ([vp, vp, vp, i64, i64, i32, vp], i32),
        "dep_projection_plan_partials": ([vp, vp, ctypes.c_size_t, P(ctypes.c_size_t)], i32),
        "dep_projection_plan_exchange": ([vp, vp, ctypes.c_size_t, P(ctypes.c_size_t)], i32),
        "dep_projection_probe_read": ([vp, ctypes.c_size_t, vp, vp], i32),
        "dep_projection_plan_selftest_exchange": ([vp, i32, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status: int, where: str):
    if status != DEP_OK:
        raise DepError(status, where)


def _ptr(t):
    """Device address of a tensor (or an int address as is)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i32_array(values):
    values = list(values)
    return (ctypes.c_int32 * max(1, len(values)))(*values), len(values)


# ---- the C functions, same names -------------------------------------------

def dep_status_string(status: int) -> str:
    return lib().dep_status_string(status).decode()


def dep_projection_version() -> int:
    return lib().dep_projection_version()


def dep_bins_index(keys, B: int) -> int:
    arr, n = _i32_array(keys)
    return lib().dep_bins_index(arr, n, B)


def dep_projection_plan(N: int, K: int, batches=(), flags: int = DEP_PLAN_DEFAULT):
    arr, n = _i32_array(batches)
    out = ctypes.c_void_p()
    _check(lib().dep_projection_plan(N, K, arr, n, flags, ctypes.byref(out)), "dep_projection_plan")
    return out.value


def dep_projection_plan_host(N: int, K: int, batches=(), sm_count: int = 152):
    arr, n = _i32_array(batches)
    out = ctypes.c_void_p()
    _check(lib().dep_projection_plan_host(N, K, arr, n, sm_count, ctypes.byref(out)),
           "dep_projection_plan_host")
    return out.value


def dep_projection_run(plan, x, W, y, B: int | None = None, stream=None) -> None:
    if B is None:
        B = x.shape[0]
    _check(lib().dep_projection_run(plan, _ptr(x), _ptr(W), _ptr(y), B, _stream(stream)),
           "dep_projection_run")


def dep_projection_run_tactic(plan, tactic: dep_tactic_t, x, W, y, B: int | None = None,
                              stream=None) -> None:
    if B is None:
        B = x.shape[0]
    _check(lib().dep_projection_run_tactic(plan, ctypes.byref(tactic), _ptr(x), _ptr(W), _ptr(y),
                                           B, _stream(stream)), "dep_projection_run_tactic")


def dep_projection_run_host(plan, x_host, W, y_host, B: int | None = None, stream=None) -> None:
    if B is None:
        B = x_host.shape[0]
    _check(lib().dep_projection_run_host(plan, _ptr(x_host), _ptr(W), _ptr(y_host), B,
                                         _stream(stream)), "dep_projection_run_host")


def dep_projection_plan_query(plan, B: int) -> dep_tactic_t:
    t = dep_tactic_t()
    _check(lib().dep_projection_plan_query(plan, B, ctypes.byref(t)), "dep_projection_plan_query")
    return t


def dep_projection_plan_table(plan) -> list:
    n = ctypes.c_int32()
    _check(lib().dep_projection_plan_table(plan, None, 0, ctypes.byref(n)), "dep_projection_plan_table")
    arr = (dep_tactic_t * max(1, n.value))()
    _check(lib().dep_projection_plan_table(plan, arr, n.value, ctypes.byref(n)),
           "dep_projection_plan_table")
    return [arr[i] for i in range(n.value)]


def dep_projection_plan_set(plan, tactic: dep_tactic_t) -> None:
    _check(lib().dep_projection_plan_set(plan, ctypes.byref(tactic)), "dep_projection_plan_set")


def dep_projection_plan_workspace(plan) -> int:
    b = ctypes.c_size_t()
    _check(lib().dep_projection_plan_workspace(plan, ctypes.byref(b)), "dep_projection_plan_workspace")
    return b.value


def dep_projection_plan_partials(plan, count: int):
    """The first `count` FP32 split-K partials of the plan's workspace (numpy)."""
    import numpy as np
    out = np.empty(count, dtype=np.float32)
    n = ctypes.c_size_t()
    _check(lib().dep_projection_plan_partials(plan, out.ctypes.data, out.nbytes, ctypes.byref(n)),
           "dep_projection_plan_partials")
    return out[: n.value // 4]


def dep_projection_plan_exchange(plan, count: int):
    """The first `count` 64-bit K-piece exchange words of the plan (numpy uint64)."""
    import numpy as np
    out = np.empty(count, dtype=np.uint64)
    n = ctypes.c_size_t()
    _check(lib().dep_projection_plan_exchange(plan, out.ctypes.data, out.nbytes, ctypes.byref(n)),
           "dep_projection_plan_exchange")
    return out[: n.value // 8]


def dep_projection_plan_save(plan, path: str) -> None:
    _check(lib().dep_projection_plan_save(plan, os.fsencode(path)), "dep_projection_plan_save")


def dep_projection_plan_load(path: str, N: int, K: int):
    out = ctypes.c_void_p()
    _check(lib().dep_projection_plan_load(os.fsencode(path), N, K, ctypes.byref(out)),
           "dep_projection_plan_load")
    return out.value


def dep_projection_plan_destroy(plan) -> None:
    lib().dep_projection_plan_destroy(plan)


def dep_projection_device_status(plan, stream=None) -> int:
    code = ctypes.c_int32()
    st = lib().dep_projection_device_status(plan, _stream(stream), ctypes.byref(code))
    if st not in (DEP_OK, DEP_ERR_TIMEOUT):
        _check(st, "dep_projection_device_status")
    return code.value


def dep_projection_selftest_timeout(limit_us: int) -> int:
    code = ctypes.c_int32()
    _check(lib().dep_projection_selftest_timeout(limit_us, ctypes.byref(code)),
           "dep_projection_selftest_timeout")
    return code.value


def dep_projection_run_static(x, W, y, N: int | None = None, K: int | None = None,
                              B: int | None = None, stream=None) -> None:
    """The no-allocation entry point (see include/dep_projection.h): for callers
    that must not allocate device memory, so cannot hold a plan."""
    if N is None:
        N, K = W.shape
    if B is None:
        B = x.shape[0]
    _check(lib().dep_projection_run_static(_ptr(x), _ptr(W), _ptr(y), N, K, B, _stream(stream)),
           "dep_projection_run_static")


def dep_projection_plan_selftest_exchange(plan, limit_us: int, stream=None) -> None:
    """Enqueue the split-K exchange's give-up self-test on the plan's workspace."""
    _check(lib().dep_projection_plan_selftest_exchange(plan, limit_us, _stream(stream)),
           "dep_projection_plan_selftest_exchange")


def dep_projection_probe_read(p, nbytes: int, sink, stream=None) -> None:
    """Read-only streaming pass over nbytes of device memory at p (measurement aid)."""
    _check(lib().dep_projection_probe_read(_ptr(p), nbytes, _ptr(sink), _stream(stream)),
           "dep_projection_probe_read")


class Projection:
    """A TP1 decode linear over one resident BF16 weight W[N,K]: the library's
    counterpart of DepProjection (runtime.dep page).  ``run(x, out)`` writes
    BF16(x . W^T) into ``out`` (allocated here when omitted) and returns it."""

    def __init__(self, weight, batches=(), flags: int = DEP_PLAN_DEFAULT):
        import torch
        if weight.dtype != torch.bfloat16 or not weight.is_cuda or not weight.is_contiguous():
            raise ValueError("weight must be a contiguous CUDA bfloat16 tensor [N, K]")
        self.weight = weight
        self.N, self.K = weight.shape
        with torch.cuda.device(weight.device):
            self.plan = dep_projection_plan(self.N, self.K, batches, flags)

    def run(self, x, out=None, stream=None):
        import torch
        if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.device != self.weight.device:
            raise ValueError("x must be a contiguous bfloat16 tensor on the weight's device")
        if out is None:
            out = torch.empty((x.shape[0], self.N), dtype=torch.bfloat16, device=x.device)
        dep_projection_run(self.plan, x, self.weight, out, x.shape[0], stream)
        return out

    def tactic(self, B: int) -> dep_tactic_t:
        return dep_projection_plan_query(self.plan, B)

    def close(self):
        if getattr(self, "plan", None):
            dep_projection_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
