"""Pins of the FP8 E4M3 cache oracle: hand-worked codes from the format
definition, a library cross-check (torch.float8_e4m3fn), and properties of the
absmax quantisation."""
import numpy as np
import pytest
import torch

from oracle import fp8


@pytest.mark.parametrize("x,code", [
    (0.0, 0x00), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (2.0 ** -9, 0x01),               # smallest subnormal
    (7 * 2.0 ** -9, 0x07),           # largest subnormal
    (2.0 ** -6, 0x08),               # smallest normal
    (0.5 * 2.0 ** -9, 0x00),         # tie between 0 and 2^-9: even -> 0
    (1.5 * 2.0 ** -9, 0x02),         # tie between codes 1 and 2: even -> 2
    (1.0625, 0x38),                  # tie between 1.0 (m=0) and 1.125 (m=1): even -> 1.0
    (1.1875, 0x3A),                  # tie between 1.125 (m=1) and 1.25 (m=2): even -> 1.25
    (1.2, 0x3A),                     # nearest is 1.25
    (464.0, 0x7E), (1e9, 0x7E),      # saturate to 448
    (240.0, 0x77),                   # 1.875 * 2^7
    (-0.25 * 2.0 ** -9, 0x80),       # rounds to zero, keeps the sign: -0
    (-0.0, 0x80),
])
def test_e4m3_hand_worked(x, code):
    assert int(fp8.e4m3_encode(np.array([x]))[0]) == code
    if abs(x) <= 448:
        assert abs(fp8.e4m3_value(np.array([code], np.uint8))[0]) <= 448


def test_e4m3_value_table():
    vals = fp8.e4m3_value(np.arange(256, dtype=np.uint8))
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    finite = vals[np.isfinite(vals)]
    assert len(finite) == 254
    # every code round-trips
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    back = fp8.e4m3_encode(fp8.e4m3_value(codes))
    assert np.array_equal(back, codes)                                  # -0 keeps its sign


def test_e4m3_matches_torch_float8():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1, 10, 100)])
    x = np.clip(x, -448, 448).astype(np.float32)
    ours = fp8.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)                                 # codes, signed zeros included


def test_quantize_rows_properties():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((64, 4, 128)) * rng.uniform(0.01, 10, (64, 4, 1))).astype(np.float32)
    x[3, 2] = 0.0                                              # an all-zero row
    codes, scales = fp8.quantize_rows(x)
    vals = fp8.e4m3_value(codes)
    amax_code = np.max(np.abs(vals), axis=-1)
    nz = scales > 0
    assert np.all(amax_code[nz] == 448.0)                      # the absmax element maps to 448
    assert scales[3, 2] == 0 and np.all(codes[3, 2] == 0)
    xh = fp8.dequantize_rows(codes, scales)
    rel = np.abs(xh - x) / np.maximum(np.max(np.abs(x), -1, keepdims=True), 1e-30)
    # E4M3 keeps 3 mantissa bits: error <= 2^-4 of |x| for normals, plus bf16 rounding
    assert np.all(np.abs(xh - x) <= np.abs(x) * (2.0 ** -4 + 2.0 ** -8) + 2.0 ** -9 * scales[..., None] * 1.01)
    assert rel.max() < 0.07
