"""Number formats and fixed-precision steps the pages prescribe — oracle.

* fp16 metadata: [vLLM-TQ] subsection "元数据为什么用 fp16 而不是 fp32" and the
  store snippets under "向量范数的存储与 norm correction 的折叠" and
  "V 的 min/max 均匀量化" convert the K norm, V scale and V zero with a plain
  fp32 -> fp16 cast, i.e. round-to-nearest-even. NumPy's float16 conversion
  is that rounding (used here as a library primitive).
* e4m3 keys: [vLLM-TQ] subsection "FP8 K 路径:不旋转,直接 cast" stores K as
  the OCP FP8 E4M3 format (e4nv: bias 7, no infinities, max finite 448). The
  encoder below is written from the format's definition: nearest representable
  value, ties to even mantissa, finite saturation at +-448.
* value quantisation: [vLLM-TQ] subsection "V 的 min/max 均匀量化" computes in
  fp32: s = (max - min) / (2^b - 1), floored at 1e-8; q = int((v - min)/s + 0.5)
  clamped to [0, 2^b - 1]. These steps decide integer codes, so the oracle
  performs them in fp32 with one IEEE rounding per operation (NumPy float32
  arithmetic), exactly as written.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "fp16_bits", "fp16_value", "e4m3_encode", "e4m3_decode_table",
    "value_quant_fp32",
]


def fp16_bits(x) -> np.ndarray:
    """Round-to-nearest-even fp16 encoding (uint16 bit patterns)."""
    return np.asarray(x).astype(np.float16).view(np.uint16)


def fp16_value(bits) -> np.ndarray:
    """float64 value of fp16 bit patterns."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def e4m3_decode_table() -> np.ndarray:
    """float64 value of each of the 256 E4M3 codes (NaN for 0x7F / 0xFF)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = e4m3_decode_table()
_E4M3_POS = _E4M3[:0x7F]            # codes 0x00..0x7E, ascending, finite


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes of float64 inputs: nearest, ties to even, saturate to +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = np.where(np.signbit(x), 0x80, 0x00)
    top = len(_E4M3_POS) - 1                       # code 0x7E = 448
    k = np.searchsorted(_E4M3_POS, np.minimum(a, _E4M3_POS[-1]), side="right") - 1
    k = np.clip(k, 0, top - 1)                     # lower neighbour code
    lo, hi = _E4M3_POS[k], _E4M3_POS[k + 1]
    down, up = a - lo, hi - a
    code = np.where(down < up, k, np.where(down > up, k + 1, np.where(k % 2 == 0, k, k + 1)))
    code = np.where(a >= _E4M3_POS[-1], top, code)
    out = (sign | code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), out).astype(np.uint8)


def value_quant_fp32(v: np.ndarray, bits: int):
    """Asymmetric uniform quantisation of each row of ``v`` in fp32.

    Returns (codes int64, scale fp32, min fp32).
    """
    v32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    levels = np.float32(2 ** bits - 1)
    mn = v32.min(axis=-1)
    mx = v32.max(axis=-1)
    s = (mx - mn) / levels
    s = np.where(s > np.float32(1e-8), s, np.float32(1e-8)).astype(np.float32)
    t = (v32 - mn[..., None]) / s[..., None] + np.float32(0.5)
    q = np.trunc(t.astype(np.float64)).astype(np.int64)
    q = np.clip(q, 0, 2 ** bits - 1)
    return q, s, mn
