"""Counter-based normal draws with bit-identical host and device forms.

Generator
---------
The word stream is SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): the i-th output of a stream
whose state starts at ``key`` is ``mix64(key + (i + 1) * GAMMA)`` (mod 2**64).
Being a pure function of ``(key, i)`` it can be evaluated for any element in
any order, on the host here and on the device in ``synth/csrc/synth_gen.cu``.

Normal approximation
--------------------
Element ``j`` of a stream takes the three words ``3j, 3j+1, 3j+2`` and sums
their twelve 16-bit fields: ``S = sum(u_i)``, ``u_i`` uniform on
``[0, 65535]``. The value is ``(S - 393210) / 65536`` which is the classic
"sum of twelve uniforms minus six" approximation of N(0, 1) (variance 1,
support [-6, 6]). Every step is integer arithmetic plus one exact scaling by
a power of two, so float32 results agree bit for bit between numpy and CUDA.

Streams
-------
``stream_key(seed, tensor, layer, seq, head)`` chains ``mix64`` over the five
indices so every (tensor, layer, sequence, KV head) segment has its own
stream; element ``j = row * head_dim + dim`` within it.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

# Tensor tags of the streams (must match synth_gen.cu).
TENSOR_K = 1
TENSOR_V = 2

_U16_SUM_MEAN = 393210  # 12 * 65535 / 2, rounded so that S - mean is symmetric


def mix64_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor: int, layer: int, seq: int, head: int) -> int:
    """64-bit key of one segment's stream."""
    k = mix64_int((seed + 1) * GAMMA)
    for idx in (tensor, layer, seq, head):
        k = mix64_int(k + (idx + 1) * GAMMA)
    return k


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def words(key: int, idx: np.ndarray) -> np.ndarray:
    """SplitMix64 outputs number ``idx`` (uint64 array) of stream ``key``."""
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx.astype(np.uint64) + np.uint64(1)) * np.uint64(GAMMA)
        return _mix64(z)


def normal12(key: int, first: int, count: int) -> np.ndarray:
    """float32 draws number ``first .. first+count-1`` of stream ``key``.

    Same words as :func:`words` (``mix64(key + (3j + t + 1) * GAMMA)``), computed
    in place to keep the host twin fast on full-size segments."""
    j = np.arange(first, first + count, dtype=np.uint64)
    s = np.zeros(count, dtype=np.uint32)
    m16 = np.uint64(0xFFFF)
    m1, m2, gamma = np.uint64(_M1), np.uint64(_M2), np.uint64(GAMMA)
    z = np.empty(count, dtype=np.uint64)
    tmp = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for t in range(3):
            np.multiply(j, np.uint64(3), out=z)
            z += np.uint64(t + 1)
            z *= gamma
            z += np.uint64(key)
            np.right_shift(z, np.uint64(30), out=tmp)
            z ^= tmp
            z *= m1
            np.right_shift(z, np.uint64(27), out=tmp)
            z ^= tmp
            z *= m2
            np.right_shift(z, np.uint64(31), out=tmp)
            z ^= tmp
            for sh in (0, 16, 32, 48):
                np.right_shift(z, np.uint64(sh), out=tmp)
                tmp &= m16
                s += tmp.astype(np.uint32)
    m = s.astype(np.int64) - _U16_SUM_MEAN
    return m.astype(np.float32) * np.float32(1.0 / 65536.0)


def segment_values(key: int, rows: int, head_dim: int, pair_scale: np.ndarray | None,
                   row_first: int = 0) -> np.ndarray:
    """float32 ``[rows, head_dim]`` block of a segment stream, rows ``row_first..``.

    ``pair_scale`` (``[head_dim // 2]`` float32, or None) multiplies both
    dimensions ``f`` and ``f + head_dim/2`` of frequency pair ``f``; the
    workloads only use exact powers of two (1 or 8), so scaling is exact.
    """
    x = normal12(key, row_first * head_dim, rows * head_dim).reshape(rows, head_dim)
    if pair_scale is not None:
        x = x * np.concatenate([pair_scale, pair_scale]).astype(np.float32)[None, :]
    return x


def to_f16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> float16 (what a cache write does)."""
    return x.astype(np.float16)


def quantize_q8_0(x: np.ndarray):
    """Quantise float32 rows ``[rows, hd]`` into planar q8_0.

    Blocks of 32 consecutive dimensions of a row share one fp16 scale
    (the ggml Q8_0 block: 32 int8 codes + one fp16 scale). Per block:
    ``d = amax / 127`` (float32, correctly rounded), stored scale
    ``fp16(d)``; code ``q = clamp(round_half_away(x / d), -127, 127)`` with
    the float32 quotient; all-zero blocks get ``d = 0, q = 0``.
    Returns ``(qs int8 [rows, hd], d float16 [rows, hd/32])``.
    """
    rows, hd = x.shape
    xb = x.reshape(rows, hd // 32, 32).astype(np.float32)
    amax = np.abs(xb).max(axis=2)
    d = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    y = (xb / safe[:, :, None]).astype(np.float32)
    y64 = y.astype(np.float64)
    q = np.sign(y64) * np.floor(np.abs(y64) + 0.5)
    q = np.clip(q, -127, 127)
    q = np.where(d[:, :, None] > 0, q, 0.0)
    return q.astype(np.int8).reshape(rows, hd), d.astype(np.float16)
