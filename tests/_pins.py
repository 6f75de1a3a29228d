"""Test-side reference helpers that are independent of the oracle.

FP8 code values come from PyTorch's float8 dtypes (a library decode), FP4
E2M1 values from the value list of the OCP MX v1.0 specification; rounding
is an exhaustive search over all codes.  Nothing here imports the
oracle or the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

E5M2, E4M3, E2M1 = 23, 24, 296
MAXV = {E4M3: 448.0, E5M2: 57344.0, E2M1: 6.0}
EMAX = {E4M3: 8, E5M2: 15, E2M1: 2}
# FLOAT4_E2M1 magnitudes of the codes 0..7 as the OCP MX v1.0 spec lists them;
# codes 8..15 are their negatives (sign bit 3)
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
_TORCH = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
_tables = {}


def fp8_table(fmt: int) -> np.ndarray:
    """float64 value of each of the 256 codes, decoded by torch (FP8), or of
    the 16 E2M1 codes from the spec's list (codes 16..255 are NaN)."""
    if fmt == E2M1 and fmt not in _tables:
        tab = np.full(256, np.nan)
        tab[:8] = E2M1_MAGNITUDES
        tab[8:16] = [-v for v in E2M1_MAGNITUDES]
        _tables[fmt] = tab
    if fmt not in _tables:
        codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        _tables[fmt] = codes.view(_TORCH[fmt]).to(torch.float64).numpy().copy()
    return _tables[fmt]


def brute_round(t: np.ndarray, fmt: int) -> np.ndarray:
    """Nearest finite FP8 code to clamp(t, -max, max) by exhaustive search;
    equal distances go to the code with an even mantissa LSB; the sign of t
    (also of a zero) is kept."""
    tab = fp8_table(fmt)
    t = np.asarray(t, dtype=np.float64).ravel()
    a = np.minimum(np.abs(t), MAXV[fmt])
    pos = np.arange(8 if fmt == E2M1 else 128)
    pos = pos[np.isfinite(tab[pos])]
    vals = tab[pos]
    out = np.empty(t.size, dtype=np.uint8)
    step = 1 << 16
    for i in range(0, t.size, step):
        d = np.abs(a[i:i + step, None] - vals[None, :])
        best = d.min(axis=1, keepdims=True)
        tie = d == best
        # among the tied codes prefer an even code (mantissa LSB 0)
        even = tie & ((pos[None, :] & 1) == 0)
        pick = np.where(even.any(axis=1), even.argmax(axis=1), tie.argmax(axis=1))
        out[i:i + step] = pos[pick]
    neg = np.signbit(t)
    out[neg] |= 0x08 if fmt == E2M1 else 0x80
    return out


def brute_mx_rows(x: np.ndarray, fmt: int):
    """MX quantisation of each row (groups of 32 along the row) with the
    element rounding done by brute_round.  The exponent is read with
    np.frexp.  Returns (codes, scale codes [rows, ceil(cols/32)])."""
    x = np.asarray(x, dtype=np.float64)
    rows, cols = x.shape
    g = (cols + 31) // 32
    pad = np.zeros((rows, g * 32))
    pad[:, :cols] = x
    blocks = pad.reshape(rows, g, 32)
    amax = np.abs(blocks).max(axis=2)
    _, e = np.frexp(amax)
    s = np.where(amax > 0, (e - 1) - EMAX[fmt], -127)
    s = np.clip(s, -127, 127)
    t = blocks * np.exp2(-s.astype(np.float64))[:, :, None]
    q = brute_round(t, fmt).reshape(rows, g * 32)[:, :cols]
    return q, (s + 127).astype(np.uint8)


def dequant_rows(q: np.ndarray, s: np.ndarray, fmt: int) -> np.ndarray:
    """value(q) * 2^(s - 127) with scale column c // 32."""
    tab = fp8_table(fmt)
    cols = q.shape[-1]
    sc = np.repeat(s[..., : (cols + 31) // 32].astype(np.float64) - 127.0, 32, axis=-1)[..., :cols]
    return tab[q] * np.exp2(sc)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
