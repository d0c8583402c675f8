"""CPU oracle for the decode projection y = BF16(x . W^T) -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product library never loads it,
and it shares no code with the CUDA path.

``linear``       exact sum, one round-to-nearest-even to BF16 (oracle.c).
``linear_rows``  the same for a subset of weight rows (sampled checks).
``mirror_fma``   bit-exact FP32 replay of the split-K FMA tactic's order (mirror.c).

Arrays are numpy ``uint16`` BF16 bit patterns, row-major and contiguous.
"""
import ctypes
import numpy as np

from . import build as _build

_lib = None


def lib():
    """Load (building if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        p16 = ctypes.POINTER(ctypes.c_uint16)
        i64 = ctypes.c_int64
        L.oracle_linear.argtypes = [p16, p16, p16, i64, i64, i64, ctypes.c_int]
        L.oracle_linear.restype = None
        L.oracle_linear_rows.argtypes = [p16, p16, ctypes.POINTER(i64), i64, p16,
                                         i64, i64, ctypes.c_int]
        L.oracle_linear_rows.restype = None
        L.oracle_max_threads.restype = ctypes.c_int
        L.mirror_fma_linear.argtypes = [p16, p16, p16, i64, i64, i64,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int]
        L.mirror_fma_linear.restype = ctypes.c_int
        _lib = L
    return _lib


def _p16(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _u16(a, shape):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    if a.shape != shape:
        raise ValueError(f"expected shape {shape}, got {a.shape}")
    return a


def linear(x, W, threads: int = 0):
    """y[B,N] = RNE_bf16(exact sum_k x[b,k] W[n,k]); x [B,K], W [N,K] uint16."""
    B, K = x.shape
    N = W.shape[0]
    x = _u16(x, (B, K))
    W = _u16(W, (N, K))
    y = np.empty((B, N), dtype=np.uint16)
    lib().oracle_linear(_p16(x), _p16(W), _p16(y), B, N, K, threads)
    return y


def linear_rows(x, W, rows, threads: int = 0):
    """y[B, len(rows)]: the oracle's outputs for weight rows ``rows`` only."""
    B, K = x.shape
    N = W.shape[0]
    x = _u16(x, (B, K))
    W = _u16(W, (N, K))
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row index out of range")
    y = np.empty((B, rows.size), dtype=np.uint16)
    lib().oracle_linear_rows(_p16(x), _p16(W),
                             rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                             rows.size, _p16(y), B, K, threads)
    return y


def mirror_fma(x, W, ctas: int, rows_per_block: int, k_tile: int = 256,
               threads: int = 0):
    """Bit-exact FP32 replay of the split-K FMA tactic for a grid of ``ctas``."""
    B, K = x.shape
    N = W.shape[0]
    x = _u16(x, (B, K))
    W = _u16(W, (N, K))
    y = np.empty((B, N), dtype=np.uint16)
    rc = lib().mirror_fma_linear(_p16(x), _p16(W), _p16(y), B, N, K, ctas,
                                 rows_per_block, k_tile, threads)
    if rc != 0:
        raise ValueError(f"mirror_fma_linear rejected its arguments ({rc})")
    return y


def max_threads() -> int:
    return lib().oracle_max_threads()
