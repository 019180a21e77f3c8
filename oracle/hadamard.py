"""Hadamard rotation of Q and K before FP8 quantisation: the oracle of the pre-pass.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages apply a Hadamard rotation to Q and K before quantising them: it roughly halves the error
that input quantisation adds and costs about 0.1% of the attention time (spbcomputers.ru ZYFA
article, FAQ "Что даёт поворот Адамара?"; captivela ZYFA article, "Angka Nyata").  Because the same
orthogonal matrix R multiplies both, (QR)(KR)^T = QK^T: attention is unchanged, while outlier
channels are spread over all channels, so the per-tensor e4m3 scale wastes less range.

Readings (the pages give no details):

* R is block-diagonal over the head dimension with normalised Walsh-Hadamard blocks H_n / sqrt(n)
  (Sylvester order), n = 128 for D = 128 and n = 64 for D = 64 and D = 192 (three blocks).
* The rotated values are computed in float32 by the radix-2 fast transform, stage h = 1, 2, 4, ...
  (butterflies a+b, a-b), then multiplied by fl32(1/sqrt(n)).
* They are quantised per tensor with the usual FP8 scale pair: scale = fl32(448 / amax) multiplies
  every value, codes = rne_e4m3_satfinite(fl32(y * scale)), and descale = fl32(amax / 448) is what
  dequantises (both 1 if amax is 0).  A multiply per element instead of a division; the codes agree
  with the division recipe except where y*scale and y/descale round to different sides of a code
  boundary (relative distance ~1e-7).
"""
from __future__ import annotations

import math

import numpy as np

from .formats import e4m3_encode_rne_satfinite

E4M3_MAX_F32 = np.float32(448.0)


def hadamard_block(d: int) -> int:
    """Hadamard block size used for head dim d."""
    if d % 128 == 0 and d // 128 == 1:
        return 128
    if d % 64 == 0:
        return 64
    raise ValueError(f"unsupported head dim {d}")


def hadamard_matrix(n: int) -> np.ndarray:
    """Sylvester-ordered Hadamard matrix of order n (entries +-1), float64."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != n:
        raise ValueError("n must be a power of two")
    return h


def fwht_f32(x, n: int) -> np.ndarray:
    """Normalised Walsh-Hadamard transform of every n-wide block of the last axis, in float32,
    radix-2 stages h = 1, 2, 4, ..., n/2, then a multiply by fl32(1/sqrt(n))."""
    y = np.array(x, dtype=np.float32, copy=True)
    shp = y.shape
    y = y.reshape(-1, shp[-1] // n, n)
    h = 1
    while h < n:
        y = y.reshape(y.shape[0], y.shape[1], n // (2 * h), 2, h)
        a = y[:, :, :, 0, :]
        b = y[:, :, :, 1, :]
        y = np.stack([a + b, a - b], axis=3)          # float32 + and -: one IEEE rounding each
        h *= 2
    y = y.reshape(shp) * np.float32(1.0 / math.sqrt(n))
    return y.astype(np.float32)


def rotate(x, d: int | None = None) -> np.ndarray:
    """x @ R in float64 with the exact block-diagonal normalised Hadamard R (reference rotation)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1] if d is None else d
    n = hadamard_block(d)
    h = hadamard_matrix(n) / math.sqrt(n)
    shp = x.shape
    return (x.reshape(-1, d // n, n) @ h).reshape(shp)


def hadamard_quantize_e4m3(x):
    """Rotate (float32 fast transform) and quantise per tensor: returns (codes uint8, descale)."""
    x = np.asarray(x)
    y = fwht_f32(x, hadamard_block(x.shape[-1]))
    amax = np.float32(np.max(np.abs(y))) if y.size else np.float32(0.0)
    descale = np.float32(amax / E4M3_MAX_F32) if amax > 0 else np.float32(1.0)
    scale = np.float32(E4M3_MAX_F32 / amax) if amax > 0 else np.float32(1.0)
    codes = e4m3_encode_rne_satfinite((y * scale).astype(np.float32).astype(np.float64))
    return codes, float(descale)
