"""Seeded synthetic inputs for relu(A·B), shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the method itself: it only draws numbers and rounds them to
fp16 once. Both sides of every parity check receive the arrays it returns.

Generator definition (counter-based, so any element can be drawn independently):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014), with the finaliser constants of Stafford's "Mix13" variant that the
  published SplitMix64 uses.  The stream with initial state ``s`` has as its e-th output
  (e = 0, 1, ...) ``mix64(s + (e + 1) * GAMMA)`` with ``GAMMA = 0x9E3779B97F4A7C15``.
* Stream keys: ``s = mix64(seed * 2**16 + tensor * 2**8 + sub)``; tensor 0 is A, 1 is B;
  ``sub`` numbers the independent draws a distribution needs (Box-Muller uses two).
* Element (r, c) of an (rows, cols) tensor is element ``e = r * cols + c`` of the stream,
  so the values never depend on a leading dimension.
* uniform[-1, 1): ``u = (x >> 40) * 2**-24``, value ``2u - 1`` (exact in float64).
* normal(0, 1): Box-Muller on ``u1 = 1 - (x1 >> 11) * 2**-53`` (in (0, 1]) and
  ``u2 = (x2 >> 11) * 2**-53``: ``sqrt(-2 ln u1) * cos(2 pi u2)``.
* Scaling happens in float64; the result is rounded once to fp16 (round to nearest even,
  numpy's float64 -> float16 conversion).
"""

from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

TENSOR_A = 0
TENSOR_B = 1


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tensor: int, sub: int = 0) -> np.uint64:
    base = (int(seed) << 16) + (int(tensor) << 8) + int(sub)
    return mix64(np.array([base & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]


def raw_u64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the SplitMix64 stream whose initial state is key."""
    e = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(key + e * GAMMA)


def _fill_chunk(out: np.ndarray, start: int, n: int, k0: np.uint64, k1: np.uint64, dist: str,
                scale: float) -> None:
    x = raw_u64(k0, start, n)
    if dist == "uniform":
        v = (x >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
        v = 2.0 * v - 1.0
    elif dist == "normal":
        x2 = raw_u64(k1, start, n)
        u1 = 1.0 - (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u2 = (x2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        v = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    elif dist == "int":
        # integers in [-2, 2]: every partial sum of a dot product stays exact in fp32
        v = ((x >> np.uint64(32)) % np.uint64(5)).astype(np.float64) - 2.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    if scale != 1.0:
        v = v * scale
    out[start:start + n] = v.astype(np.float16)


def _fill(rows: int, cols: int, seed: int, tensor: int, dist: str, scale: float) -> np.ndarray:
    if dist not in ("uniform", "normal", "int"):
        raise ValueError(f"unknown distribution {dist!r}")
    total = rows * cols
    out = np.empty(total, dtype=np.float16)
    k0 = stream_key(seed, tensor, 0)
    k1 = stream_key(seed, tensor, 1)
    starts = list(range(0, total, _CHUNK))
    if len(starts) <= 1:
        for start in starts:
            _fill_chunk(out, start, min(_CHUNK, total - start), k0, k1, dist, scale)
    else:
        # chunks are independent slices of the counter-based stream: drawing them on several
        # threads (numpy releases the GIL in these loops) gives the same values as in order
        import concurrent.futures as cf
        import os

        workers = min(len(starts), os.cpu_count() or 1, 16)
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(lambda st: _fill_chunk(out, st, min(_CHUNK, total - st), k0, k1, dist,
                                               scale), starts))
    return out.reshape(rows, cols)


def tensor(rows: int, cols: int, seed: int, tensor_id: int, dist: str = "uniform",
           scale: float = 1.0) -> np.ndarray:
    """A (rows, cols) row-major fp16 array drawn as described in the module docstring."""
    if rows < 0 or cols < 0:
        raise ValueError("negative shape")
    return _fill(int(rows), int(cols), int(seed), int(tensor_id), dist, float(scale))


def embed(x: np.ndarray, ld: int, fill: float = 0.0) -> np.ndarray:
    """Copy (rows, cols) into a (rows, ld) buffer; returns the padded buffer (rows*ld elements)."""
    rows, cols = x.shape
    if ld < cols:
        raise ValueError("ld < cols")
    buf = np.full((rows, ld), fill, dtype=x.dtype)
    buf[:, :cols] = x
    return buf


def int4_weights(K: int, N: int, seed: int, ldq: int | None = None) -> np.ndarray:
    """Packed 4-bit weights: K rows of ldq (>= ceil(N/8)) uint32 words; nibble e of word c is
    column 8c+e, each nibble uniform in [0, 15] from the stream (seed, tensor 2); words past
    ceil(N/8) and nibbles past column N are zero."""
    words = (N + 7) // 8
    ldq = words if ldq is None else ldq
    if ldq < words:
        raise ValueError("ldq < ceil(N/8)")
    k0 = stream_key(seed, 2, 0)
    out = np.zeros((K, ldq), dtype=np.uint32)
    nib = np.empty((K, words * 8), dtype=np.uint32)
    flat = (raw_u64(k0, 0, K * N) >> np.uint64(60)).astype(np.uint32).reshape(K, N)
    nib[:, :N] = flat
    nib[:, N:] = 0
    nib = nib.reshape(K, words, 8)
    packed = np.zeros((K, words), dtype=np.uint32)
    for e in range(8):
        packed |= nib[:, :, e] << np.uint32(4 * e)
    out[:, :words] = packed
    return out


def int4_scales(groups: int, N: int, seed: int, scale: float, lds: int | None = None) -> np.ndarray:
    """fp16 group scales, groups x lds (>= N): uniform in [0.5, 1.5) x scale, rounded once."""
    lds = N if lds is None else lds
    s = tensor(groups, N, seed, 3, "uniform", 1.0).astype(np.float64) * 0.5 + 1.0
    out = np.zeros((groups, lds), dtype=np.float16)
    out[:, :N] = (s * scale).astype(np.float16)
    return out
