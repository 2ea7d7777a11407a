"""Seeded synthetic inputs for the benchmark workloads.

Holds none of the quantized-matmul arithmetic: it only draws numbers.  The
same arrays feed the CPU oracle and the CUDA library.

Generator: SplitMix64 in counter form.  The i-th 64-bit output of stream
``seed`` is ``mix(seed + (i + 1) * 0x9E3779B97F4A7C15)`` (mod 2^64), with the
published SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Uniforms in (0, 1] are
``((z >> 11) + 1) * 2^-53``.  Normals come from Box-Muller in double
precision on consecutive uniform pairs: normal ``2p`` is ``r*cos(2*pi*u2)`` and
normal ``2p+1`` is ``r*sin(2*pi*u2)`` with ``r = sqrt(-2 ln u1)``, ``u1``/``u2``
the uniforms ``2p``/``2p+1``.  The value returned is ``float32(sigma * z)``.

Each workload draws from one stream per seed, in this order: weights
row-major [N, K], then activations [m, K], then the extras (outlier mask,
ternary values, the absmean draw), each from its own counter range.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of SplitMix64 stream ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        return _mix(np.uint64(seed & (2**64 - 1)) + idx * _GAMMA)


def uniform(seed: int, start: int, count: int) -> np.ndarray:
    """float64 uniforms in (0, 1] from outputs start .. start+count-1."""
    z = raw_u64(seed, start, count)
    return ((z >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * (2.0 ** -53)


def _normal_chunk(seed: int, start: int, count: int, sigma: float) -> np.ndarray:
    # normals start..start+count-1; normal i uses uniforms 2*(i//2), 2*(i//2)+1
    p0 = start // 2
    p1 = (start + count + 1) // 2
    u = uniform(seed, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    r = np.sqrt(-2.0 * np.log(u[:, 0]))
    th = (2.0 * np.pi) * u[:, 1]
    z = np.empty((p1 - p0, 2), np.float64)
    z[:, 0] = r * np.cos(th)
    z[:, 1] = r * np.sin(th)
    z = z.ravel()[start - 2 * p0: start - 2 * p0 + count]
    return (sigma * z).astype(np.float32)


def normal(seed: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """float32 N(0, sigma^2) values ``start .. start+count-1`` of stream ``seed``.

    Normal index i consumes uniforms 2*(i//2) and 2*(i//2)+1, so a stream of
    normals occupies the uniform counters [2*start, 2*(start+count))."""
    out = np.empty(count, np.float32)
    spans = [(s, min(_CHUNK, count - s)) for s in range(0, count, _CHUNK)]

    def work(span):
        s, c = span
        out[s:s + c] = _normal_chunk(seed, start + s, c, sigma)

    if len(spans) <= 1:
        for sp in spans:
            work(sp)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(work, spans))
    return out


def ternary(seed: int, start: int, count: int) -> np.ndarray:
    """int8 values iid uniform on {-1, 0, +1}: floor(3 * (1 - u)) - 1."""
    out = np.empty(count, np.int8)
    for s in range(0, count, _CHUNK):
        c = min(_CHUNK, count - s)
        u = uniform(seed, start + s, c)
        out[s:s + c] = (np.floor(3.0 * (1.0 - u)).astype(np.int64) - 1).clip(-1, 1).astype(np.int8)
    return out


class Stream:
    """Sequential reader over one seed's SplitMix64 stream (uniform counters)."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0  # next uniform counter

    def normal(self, shape, sigma: float = 1.0) -> np.ndarray:
        count = int(np.prod(shape))
        start = (self.pos + 1) // 2
        a = normal(self.seed, start, count, sigma)
        self.pos = 2 * (start + count)
        return a.reshape(shape)

    def uniform(self, shape) -> np.ndarray:
        count = int(np.prod(shape))
        a = uniform(self.seed, self.pos, count)
        self.pos += count
        return a.reshape(shape)

    def ternary(self, shape) -> np.ndarray:
        count = int(np.prod(shape))
        a = ternary(self.seed, self.pos, count)
        self.pos += count
        return a.reshape(shape)


# --------------------------------------------------------------------------
# The benchmark workloads as concrete seeded inputs.

LAYER_SET_7B = [(4096, 4096)] * 4 + [(11008, 4096)] * 2 + [(4096, 11008)]  # (N, K)


def q4_0_case(seed: int, n: int, k: int, m: int, w_sigma: float = 0.02,
              outlier_p: float = 0.0, outlier_mult: float = 20.0):
    """Weights f32 [n, k] ~ N(0, w_sigma^2), activations f32 [m, k] ~ N(0, 1);
    optionally each activation independently multiplied by ``outlier_mult``
    with probability ``outlier_p``."""
    st = Stream(seed)
    w = st.normal((n, k), w_sigma)
    x = st.normal((m, k), 1.0)
    if outlier_p > 0.0:
        u = st.uniform((m, k))
        x = np.where(u <= outlier_p, x * np.float32(outlier_mult), x).astype(np.float32)
    return w, x


def bitnet_case(seed: int, n: int, k: int, m: int, absmean_sigma: float = 0.02):
    """Ternary weights int8 [n, k] iid uniform on {-1,0,1}; activations f32
    [m, k] ~ N(0,1); the per-tensor weight scale is mean|v| over an
    independent f32 N(0, absmean_sigma^2) draw of n*k values (accumulated in
    double, rounded once to f32)."""
    st = Stream(seed)
    t = st.ternary((n, k))
    x = st.normal((m, k), 1.0)
    v = st.normal((n * k,), absmean_sigma)
    absmean = np.float32(np.abs(v.astype(np.float64)).mean())
    return t, x, float(absmean)
