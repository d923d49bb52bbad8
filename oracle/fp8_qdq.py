"""FP8 (E4M3) state quantize-dequantize oracle: TEST INFRASTRUCTURE ONLY.

Statement of the state quantizer of the "linear_attention.reference" page (its FP8 state
entry): dynamic E4M3 quantize-dequantize with one scale per [Dk, block_v] tile of a key-first
state [..., Dk, Dv]; an all-zero tile uses scale one; a partial last tile of value columns is
a tile of its own; scales and rounding carry no derivative (the gradient passes unchanged).

Readings (the page prints no formula): scale = amax / 448 over the tile (448, the largest
finite E4M3 value), or 1 when amax is 0; the stored code is x / scale rounded to the nearest
E4M3 value (ties to even mantissa), saturating at +-448; the result is code * scale.  The
scale and the division are taken in float32, the dtype of the states, so that the code the
rounding picks is the same on the GPU (where a quantised code is decided, both sides decide it
in the same precision).  E4M3 is decoded here from its definition: sign, 4 exponent bits with
bias 7, 3 mantissa bits; exponent 0 holds the subnormals m / 8 * 2^-6; the all-ones pattern
S.1111.111 is NaN and there is no infinity, so the finite values run to 1.75 * 2^8 = 448.

Pinned in ``tests/test_fp8_qdq_oracle.py`` (every code of the format, ties, saturation, the
zero tile, partial tiles, idempotence, and torch's float8_e4m3fn cast as a second opinion).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Every finite E4M3 value of the 256 codes (the two NaNs dropped, +-0 merged), ascending,
    from the format's definition."""
    vals = []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue  # NaN
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
    return np.unique(np.array(vals, dtype=np.float64))


_POS = e4m3_values()
_POS = _POS[_POS >= 0.0]          # 0, subnormals, normals up to 448


def _is_even_code(v: float) -> bool:
    """True when the E4M3 code of the non-negative value v has an even mantissa field."""
    if v == 0.0:
        return True
    e = int(np.floor(np.log2(v)))
    if e < -6:  # subnormal: v = m / 8 * 2^-6
        m = int(round(v / 2.0 ** -9))
    else:
        m = int(round((v / 2.0 ** e - 1.0) * 8.0))
    return m % 2 == 0


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Rounds every value to the nearest finite E4M3 value, ties to the even mantissa, with
    saturation at +-448.  Exact for float32 or float64 input (the grid is exact in double)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(_POS, a)               # _POS[idx - 1] < a <= _POS[idx]
    idx = np.clip(idx, 1, len(_POS) - 1)
    lo, hi = _POS[idx - 1], _POS[idx]
    out = np.where(a - lo < hi - a, lo, hi)
    tie = (a - lo) == (hi - a)
    if np.any(tie):
        for k in zip(*np.nonzero(tie)):
            out[k] = lo[k] if _is_even_code(lo[k]) else hi[k]
    out = np.where(a == 0.0, 0.0, out)
    return np.copysign(out, x)


def state_fp8_qdq(state: np.ndarray, block_v: int = 64) -> np.ndarray:
    """Quantize-dequantize of key-first states [..., Dk, Dv], one scale per [Dk, block_v]
    tile.  Returns float32 (the states' dtype)."""
    st = np.asarray(state, dtype=np.float32)
    Dv = st.shape[-1]
    out = np.empty_like(st)
    for v0 in range(0, Dv, block_v):
        t = st[..., v0:v0 + block_v]
        amax = np.max(np.abs(t), axis=(-2, -1), keepdims=True).astype(np.float32)
        scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        code = round_e4m3((t / scale).astype(np.float32))
        out[..., v0:v0 + block_v] = (code.astype(np.float32) * scale).astype(np.float32)
    return out
