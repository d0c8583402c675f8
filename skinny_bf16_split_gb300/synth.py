"""Seeded synthetic inputs for the decode projection (no method arithmetic here).

Both the CUDA path's tests/benchmark and the CPU oracle take their inputs from
this module, and from nothing else, so that the two sides see identical bits.

Generator (counter based, so any element can be made without the ones before):
  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): output n of the stream with key k is
    mix64(k + (n + 1) * 0x9E3779B97F4A7C15), and the key of (seed, tensor) is
    mix64((seed << 32) | tensor).
  * Two 53-bit uniforms per pair of elements, u = (r >> 11) * 2^-53, and the
    Box-Muller transform in float64: rad = sqrt(-2 ln(1 - u1)), angle = 2 pi u2,
    element 2i = rad cos(angle), element 2i+1 = rad sin(angle).
  * Scaled by sigma, then rounded once from float64 to BF16 (nearest, ties to
    even).  The bits depend on the platform's float64 log/sin/cos only through
    the last bit of the float64 value, so they agree between machines except in
    the rare case where that bit decides a BF16 rounding.

Workloads (the shapes the runtime.dep page names for one DSA/KDA layer at TP1:
DSA packed input projection 14560 x 7168, o_proj 7168 x 12288, KDA packed input
projection 49376 x 7168; batches are decode rows).  W ~ N(0, 0.02); x ~ N(0, 1),
and for the DSA B=1 case each x row is scaled to unit RMS, as the attention
layers receive normalised rows (runtime.dep page, DepAttention.run_wide).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids inside one seed's stream
W_ID, X_ID = 1, 2


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([(int(seed) << 32) | int(tensor)], dtype=np.uint64)
        return _mix64(k)[0]


def _normals_pairs(key: np.uint64, p0: int, p1: int) -> np.ndarray:
    """float64 normals for elements [2 p0, 2 p1) of the stream `key`."""
    with np.errstate(over="ignore"):
        n = np.arange(2 * p0, 2 * p1, dtype=np.uint64)
        r = _mix64(key + (n + np.uint64(1)) * _GOLDEN)
    u = (r >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log1p(-u1))
    ang = (2.0 * np.pi) * u2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)
    out[0::2] = rad * np.cos(ang)
    out[1::2] = rad * np.sin(ang)
    return out


def bf16_from_f64(v: np.ndarray) -> np.ndarray:
    """Round float64 values once to BF16 bit patterns (nearest, ties to even)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint16)
    sign = np.signbit(v).astype(np.uint16) << np.uint16(15)
    a = np.abs(v)
    nan = np.isnan(v)
    inf = np.isinf(v)
    fin = ~(nan | inf) & (a > 0)
    m, ex = np.frexp(np.where(fin, a, 1.0))  # a = m 2^ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1               # a in [2^e, 2^(e+1))
    normal = fin & (e >= -126)
    # normal: 8 significant bits, M = rint(a / 2^(e-7)) in [128, 256]
    M = np.rint(np.ldexp(np.where(fin, a, 0.0), (7 - e).astype(np.int32)))
    carry = normal & (M == 256)
    e = np.where(carry, e + 1, e)
    M = np.where(carry, 128, M)
    field = e + 127
    over = normal & (field >= 255)
    enc_n = (field.clip(0, 254) << 7) | (M.astype(np.int64).clip(128, 255) - 128)
    # subnormal: fixed quantum 2^-133, M = rint(a * 2^133) in [0, 128]
    Ms = np.rint(np.ldexp(np.where(fin & ~normal, a, 0.0), 133)).astype(np.int64)
    out = np.where(normal, enc_n, Ms).astype(np.uint16)
    out = np.where(over | inf, np.uint16(0x7F80), out)
    out = np.where(nan, np.uint16(0x7FC0), out | sign)
    return out.astype(np.uint16)


def _chunks(total: int, parts: int):
    step = max(1, -(-total // parts))
    return [(i, min(total, i + step)) for i in range(0, total, step)]


def normal_f64(seed: int, tensor: int, count: int, threads: int | None = None) -> np.ndarray:
    """`count` float64 N(0,1) values of stream (seed, tensor)."""
    key = _key(seed, tensor)
    pairs = (count + 1) // 2
    threads = threads or os.cpu_count() or 1
    spans = _chunks(pairs, max(1, min(threads * 4, pairs // 65536 + 1)))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda s: _normals_pairs(key, *s), spans))
    out = np.concatenate(parts) if parts else np.empty(0)
    return out[:count]


def normal_bf16(seed: int, tensor: int, shape, sigma: float = 1.0,
                threads: int | None = None) -> np.ndarray:
    """BF16 bits of N(0, sigma^2) values, shape `shape`, stream (seed, tensor)."""
    shape = tuple(int(s) for s in shape)
    count = int(np.prod(shape)) if shape else 1
    key = _key(seed, tensor)
    pairs = (count + 1) // 2
    threads = threads or os.cpu_count() or 1
    out = np.empty(2 * pairs, dtype=np.uint16)

    def work(span):
        p0, p1 = span
        out[2 * p0:2 * p1] = bf16_from_f64(_normals_pairs(key, p0, p1) * sigma)

    spans = _chunks(pairs, max(1, min(threads * 4, pairs // 65536 + 1)))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(work, spans))
    return out[:count].reshape(shape)


def normal_bf16_head(seed: int, tensor: int, shape, rows: int, sigma: float = 1.0) -> np.ndarray:
    """The first `rows` rows of normal_bf16(seed, tensor, shape, sigma), bit for
    bit, without generating the rest (the stream is counter-based: element n of
    a row-major tensor depends only on n)."""
    shape = tuple(int(s) for s in shape)
    cols = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    rows = max(0, min(int(rows), shape[0]))
    count = rows * cols
    pairs = (count + 1) // 2
    vals = bf16_from_f64(_normals_pairs(_key(seed, tensor), 0, pairs) * sigma) if pairs else np.empty(0, np.uint16)
    return vals[:count].reshape((rows,) + shape[1:])


def rms_rows_bf16(seed: int, tensor: int, shape) -> np.ndarray:
    """BF16 bits of N(0,1) rows each scaled (in float64) to unit RMS."""
    rows, cols = (int(s) for s in shape)
    z = normal_f64(seed, tensor, rows * cols).reshape(rows, cols)
    rms = np.sqrt(np.mean(z * z, axis=1, keepdims=True))
    return bf16_from_f64(z / rms)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """BF16 bits -> float32 values (exact: BF16 is the top half of FP32)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --- the workloads ----------------------------------------------------------

DSA = (14560, 7168)     # packed [q_a | kv_a | gate | wk | wv] input projection
OPROJ = (7168, 12288)   # o_proj: 96 heads x 128 -> 7168
KDA = (49376, 7168)     # packed KDA input projection


@dataclass(frozen=True)
class Call:
    """One projection call y[B,N] = x[B,K] W[N,K]^T of a workload."""
    name: str
    N: int
    K: int
    B: int
    seed: int
    w_id: int = W_ID
    x_id: int = X_ID
    x_rms: bool = False

    def weight(self) -> np.ndarray:
        return normal_bf16(self.seed, self.w_id, (self.N, self.K), sigma=0.02)

    def weight_head(self, rows: int) -> np.ndarray:
        """The first `rows` rows of weight() (for sampled CPU work)."""
        return normal_bf16_head(self.seed, self.w_id, (self.N, self.K), rows, sigma=0.02)

    def activations(self) -> np.ndarray:
        if self.x_rms:
            return rms_rows_bf16(self.seed, self.x_id, (self.B, self.K))
        return normal_bf16(self.seed, self.x_id, (self.B, self.K))

    @property
    def algorithmic_bytes(self) -> int:
        """W + x + y bytes: what one call must move at least once."""
        return 2 * (self.N * self.K + self.B * self.K + self.B * self.N)

    @property
    def weight_key(self):
        return (self.N, self.K, self.seed, self.w_id)


def workload(name: str) -> list[Call]:
    """The calls of one named workload, in order."""
    if name == "dsa_b1":
        return [Call("dsa_b1", *DSA, B=1, seed=0, x_rms=True)]
    if name == "oproj_sweep":
        return [Call(f"oproj_b{b}", *OPROJ, B=b, seed=s)
                for s, b in enumerate((1, 2, 4, 8, 16))]
    if name == "kda_sweep":
        return [Call(f"kda_b{b}", *KDA, B=b, seed=s) for s, b in enumerate((1, 4, 8, 16))]
    if name == "dsa_wide":
        return [Call(f"dsa_b{b}", *DSA, B=b, seed=s) for s, b in enumerate((32, 64, 128, 256))]
    if name == "dsa_verify":
        # speculative verify steps: B = requests x q tokens (q = 2..4)
        return [Call(f"dsa_verify_b{b}", *DSA, B=b, seed=s) for s, b in enumerate((3, 6, 12, 24, 48))]
    if name == "tp_sharded":
        # one rank's share of a TP-G hybrid step: input projection rows N/G,
        # o_proj reduction K/G (the all-reduce of the partials is a separate step)
        calls = []
        for s, g in enumerate((2, 4, 8)):
            calls.append(Call(f"dsa_tp{g}", DSA[0] // g, DSA[1], B=16, seed=s))
        for s, g in enumerate((2, 4, 8)):
            calls.append(Call(f"oproj_tp{g}", OPROJ[0], OPROJ[1] // g, B=16, seed=3 + s))
        return calls
    if name == "baseline":
        # the five configurations of the decode-projection benchmark in one step:
        # DSA B=1, the o_proj sweep, the KDA sweep, wide DSA batches, the chain
        return [c for part in ("dsa_b1", "oproj_sweep", "kda_sweep", "dsa_wide", "chain") for c in workload(part)]
    if name == "chain":
        calls = []
        for layer in range(8):
            base = 16 + 4 * layer
            calls.append(Call(f"chain_l{layer}_dsa", *DSA, B=16, seed=7, w_id=base, x_id=base + 2))
            calls.append(Call(f"chain_l{layer}_oproj", *OPROJ, B=16, seed=7, w_id=base + 1,
                              x_id=base + 3))
        return calls
    raise KeyError(f"unknown workload {name!r}")


WORKLOADS = ("baseline", "dsa_b1", "oproj_sweep", "kda_sweep", "dsa_wide", "chain", "dsa_verify", "tp_sharded")
