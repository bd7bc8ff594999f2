"""CPU oracle for the FP8 E4M3 prefix cache (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the CUDA path never does.

Source: "Qwen-Image 2.1 deployment notes" (10100.com), prefix-KV-cache
section: the prefix cache is quantised to FP8 E4M3 with one FP32 scale per
token and attention head, in two modes (K and V, or V only; V only keeps K in
bf16).  The pages do not say how the scale is chosen; the reading used here
(listed in the design notes) is absmax scaling of each 128-value (token, head)
row onto the E4M3 range, all arithmetic in fp32:

    amax  = max |x|                                  (x is the bf16 row)
    scale = amax / 448            (fp32 division; 0 for an all-zero row)
    code  = E4M3(x * (448 / amax)) round-to-nearest-even, saturating at +-448
    x_hat = bf16(fp32(value(code)) * scale)          (dequantised key/value)

E4M3 (the OCP 8-bit float "E4M3FN"): 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no infinities;
S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_value(code) -> np.ndarray:
    """Value of E4M3 codes (uint8 array) as float64 (NaN for the NaN codes)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def _all_finite_values():
    codes = np.arange(0x80, dtype=np.uint8)              # non-negative codes
    vals = e4m3_value(codes)
    keep = np.isfinite(vals)
    return codes[keep], vals[keep]                        # sorted ascending by construction


_POS_CODES, _POS_VALS = _all_finite_values()


def e4m3_encode(x) -> np.ndarray:
    """Round float values to E4M3 codes: nearest, ties to the even code
    (mantissa LSB 0), magnitudes above 448 saturate to 448, the sign is kept
    (negative values that round to zero give -0, code 0x80), NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    mag = np.minimum(np.abs(x), E4M3_MAX)
    # index of the largest representable value <= mag
    lo = np.clip(np.searchsorted(_POS_VALS, mag, side="right") - 1, 0, len(_POS_VALS) - 1)
    hi = np.minimum(lo + 1, len(_POS_VALS) - 1)
    d_lo = mag - _POS_VALS[lo]
    d_hi = _POS_VALS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[lo] & 1 == 1) & (hi != lo))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    # rounding keeps the sign, also for a value that rounds to zero (-0 = 0x80)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), np.uint8(0x7F), code)
    out[...] = code
    return out


def _bf16_round(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even), returned as float32."""
    b = np.asarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Absmax E4M3 quantisation of rows along the last axis (fp32 arithmetic).

    Returns (codes uint8, same shape; scales float32, shape[:-1])."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    inv = np.where(amax > 0, np.float32(E4M3_MAX) / np.where(amax > 0, amax, 1), 0).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


def dequantize_rows(codes, scales) -> np.ndarray:
    """x_hat = bf16(fp32(value(code)) * scale), as float32 values."""
    v = e4m3_value(codes).astype(np.float32)
    prod = (v * np.asarray(scales, dtype=np.float32)[..., None]).astype(np.float32)
    return _bf16_round(prod)


def cache_append_fp8(k, v, cu_seqlens_k, cu_prefix, mode: str, layer: int, caches: dict):
    """Clone each sequence's prefix into the quantised cache of one layer.

    ``caches`` holds NumPy arrays ``k`` (bf16 bits as uint16 in "v" mode, E4M3
    codes in "kv" mode), ``v`` (E4M3 codes), ``sk``/``sv`` (float32 scales),
    shaped ``[L][H][cap][128]`` / ``[L][H][cap]``; updated in place.
    """
    if hasattr(k, "detach"):
        kb = k.detach().cpu().contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        kf = k.detach().cpu().float().numpy()
        vf = v.detach().cpu().float().numpy()
    else:
        raise TypeError("k and v must be bf16 torch tensors")
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    cp = np.asarray(cu_prefix, dtype=np.int64)
    for b in range(len(ck) - 1):
        n = cp[b + 1] - cp[b]
        src = slice(ck[b], ck[b] + n)
        dst = slice(cp[b], cp[b] + n)
        vc, vs = quantize_rows(vf[src])                 # [n, H, 128], [n, H]
        caches["v"][layer, :, dst] = np.transpose(vc, (1, 0, 2))
        caches["sv"][layer, :, dst] = vs.T
        if mode == "kv":
            kc, ks = quantize_rows(kf[src])
            caches["k"][layer, :, dst] = np.transpose(kc, (1, 0, 2))
            caches["sk"][layer, :, dst] = ks.T
        else:
            caches["k"][layer, :, dst] = np.transpose(kb[src], (1, 0, 2))
    return caches
