"""Pins of the FP8 E4M3 cache oracle: hand-worked codes from the format
definition, a library cross-check (torch.float8_e4m3fn), properties of the
absmax quantisation, hand-worked bf16 rounding of the dequantised values (and a
torch bfloat16 cross-check), a hand-indexed layout of the quantising append in
both modes, and planted mistakes that each fail one of these pins."""
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


# ---- bf16 rounding of the dequantised value ------------------------------------------
# Hand-worked from the bf16 format (the upper 16 bits of an IEEE binary32, rounded to
# nearest with ties to the even upper half): fp32 bits in, bf16 bits out.
BF16_CASES = [
    (0x3F808000, 0x3F80),   # 1 + 2^-8: half-way between 0x3F80 and 0x3F81, tie to even (down)
    (0x3F818000, 0x3F82),   # 1 + 3*2^-8: half-way between 0x3F81 and 0x3F82, tie to even (up)
    (0x3F808001, 0x3F81),   # just above half-way: up
    (0x3F807FFF, 0x3F80),   # just below half-way: down
    (0xBF818000, 0xBF82),   # negative tie: the magnitude rounds to even
    (0x3F7FFFFF, 0x3F80),   # 0.99999994: the carry moves into the exponent, giving 1.0
    (0x00018000, 0x0002),   # subnormal tie, odd lower half: up
    (0x3F800000, 0x3F80),   # exact values stay
]


def _f32(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def pin_bf16_round_hand_worked(mod):
    got = mod._bf16_round(_f32([b for b, _ in BF16_CASES])).view(np.uint32)
    for (b, want), g in zip(BF16_CASES, got):
        assert g & 0xFFFF == 0, hex(b)
        assert g >> 16 == want, (hex(b), hex(g >> 16), hex(want))


def pin_bf16_round_matches_torch(mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(50000).astype(np.float32) * np.float32(3.0),
        _f32(rng.integers(0, 2 ** 32, 50000, dtype=np.uint64).astype(np.uint32)),
    ])
    x = x[np.isfinite(x) & (np.abs(x) < np.float32(3e38))]
    ours = mod._bf16_round(x).view(np.uint32) >> 16
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours.astype(np.uint16), theirs)


def pin_dequantize_hand_worked(mod):
    """x_hat = bf16(value(code) * scale): products chosen to land on and beside bf16 ties."""
    cases = [
        (0x38, 1.0 + 2.0 ** -8, 1.0),                        # 1.0 * (1 + 2^-8): tie, down to 1.0
        (0x38, 1.0 + 3 * 2.0 ** -8, 1.015625),               # tie, up to 1 + 2^-6
        (0x38, 1.0 + 2.0 ** -8 + 2.0 ** -20, 1.0078125),     # above half-way
        (0xB8, 1.0 + 3 * 2.0 ** -8, -1.015625),              # -1.0: negative tie
        (0x3A, 0.5, 0.625),                                  # 1.25 * 0.5, exact
        (0x7E, 2.0 ** -8, 1.75),                             # 448 * 2^-8, exact
        (0x01, 2.0 ** 9, 1.0),                               # smallest subnormal 2^-9 * 2^9
    ]
    for code, scale, want in cases:
        got = mod.dequantize_rows(np.array([[code]], dtype=np.uint8), np.array([scale], np.float32))
        assert got.dtype == np.float32 and got[0, 0] == np.float32(want), (hex(code), scale, got)


# ---- the quantising append: which row goes where -------------------------------------
def _layout_inputs():
    """Two sequences whose cache offsets differ from their key offsets.

    Row (token t, head h) of K is [a, -a, a/2, 0, ...] with a = 1 + t + 13 h, of V the
    same with a = 100 + t + 13 h: every value is exact in bf16, the row's absmax is a,
    so its codes are [448, -448, 224, 0, ...] = [0x7E, 0xFE, 0x76, 0, ...] and its
    scale a / 448 names the source row."""
    T, H = 12, 3
    a_k = (1 + np.arange(T)[:, None] + 13 * np.arange(H)[None, :]).astype(np.float32)
    a_v = a_k + 99
    def rows(a):
        x = np.zeros((T, H, 128), dtype=np.float32)
        x[:, :, 0], x[:, :, 1], x[:, :, 2] = a, -a, a / 2
        return torch.from_numpy(x).to(torch.bfloat16)
    k, v = rows(a_k), rows(a_v)
    cu_k = np.array([0, 5, 12])
    cu_p = np.array([0, 3, 9])      # prefixes of 3 and 6 tokens; sequence 1 starts at key 5
    return k, v, cu_k, cu_p, a_k, a_v


def _empty_caches(mode, layers=2, H=3, cap=11):
    kdt = np.uint8 if mode == "kv" else np.uint16
    return {
        "k": np.full((layers, H, cap, 128), 0x55, dtype=kdt),
        "v": np.full((layers, H, cap, 128), 0x55, dtype=np.uint8),
        "sk": np.full((layers, H, cap), -1.0, dtype=np.float32),
        "sv": np.full((layers, H, cap), -1.0, dtype=np.float32),
    }


def _expected_code_row():
    r = np.zeros(128, dtype=np.uint8)
    r[0], r[1], r[2] = 0x7E, 0xFE, 0x76
    return r


# cache row c of the layer <- key row src (sequence 0: tokens 0..2; sequence 1: keys 5..10)
_LAYOUT = list(zip(range(9), [0, 1, 2, 5, 6, 7, 8, 9, 10]))


def pin_append_fp8_layout(mod):
    for mode in ("v", "kv"):
        k, v, cu_k, cu_p, a_k, a_v = _layout_inputs()
        caches = mod.cache_append_fp8(k, v, cu_k, cu_p, mode, 1, _empty_caches(mode))
        kbits = k.view(torch.int16).numpy().view(np.uint16)
        for h in range(3):
            for c, src in _LAYOUT:
                assert np.array_equal(caches["v"][1, h, c], _expected_code_row()), (mode, h, c)
                assert caches["sv"][1, h, c] == np.float32(a_v[src, h]) / np.float32(448), (mode, h, c)
                if mode == "kv":
                    assert np.array_equal(caches["k"][1, h, c], _expected_code_row()), (h, c)
                    assert caches["sk"][1, h, c] == np.float32(a_k[src, h]) / np.float32(448), (h, c)
                else:   # V only: K is the bf16 row itself
                    assert np.array_equal(caches["k"][1, h, c], kbits[src, h]), (h, c)
        # nothing else is written: the other layer, the rows past the prefixes, unused scales
        assert np.all(caches["v"][0] == 0x55) and np.all(caches["v"][1, :, 9:] == 0x55)
        assert np.all(caches["k"][0] == 0x55) and np.all(caches["k"][1, :, 9:] == 0x55)
        assert np.all(caches["sv"][0] == -1) and np.all(caches["sv"][1, :, 9:] == -1)
        if mode == "v":
            assert np.all(caches["sk"] == -1)


FP8_PINS = [pin_bf16_round_hand_worked, pin_bf16_round_matches_torch, pin_dequantize_hand_worked,
            pin_append_fp8_layout]


def test_fp8_pins_hold():
    for pin in FP8_PINS:
        pin(fp8)


# ---- planted mistakes: each must fail at least one pin --------------------------------
_real_append = fp8.cache_append_fp8
_real_quantize = fp8.quantize_rows


def _truncating_bf16(x32):
    b = np.asarray(x32, dtype=np.float32).view(np.uint32)
    return ((b >> 16) << 16).astype(np.uint32).view(np.float32)


def _append_cache_rows_at_key_offsets(k, v, cu_seqlens_k, cu_prefix, mode, layer, caches):
    """The append with the destination taken from cu_seqlens_k instead of cu_prefix."""
    ck = np.asarray(cu_seqlens_k, dtype=np.int64)
    cp = np.asarray(cu_prefix, dtype=np.int64)
    fake_cp = cp.copy()
    for b in range(len(ck) - 1):
        fake_cp[b] = ck[b]
        fake_cp[b + 1] = ck[b] + (cp[b + 1] - cp[b])
        _real_append(k, v, ck[b:b + 2], fake_cp[b:b + 2], mode, layer, caches)
    return caches


def _scale_inverted(x):
    codes, scale = _real_quantize(x)
    with np.errstate(divide="ignore"):
        inv = np.where(scale > 0, np.float32(1.0) / np.where(scale > 0, scale, 1), 0)
    return codes, inv.astype(np.float32)


FP8_MUTANTS = {
    "bf16_truncation": ("_bf16_round", _truncating_bf16),
    "append_at_key_offsets": ("cache_append_fp8", _append_cache_rows_at_key_offsets),
    "k_and_v_swapped": ("cache_append_fp8",
                        lambda k, v, *a, **kw: _real_append(v, k, *a, **kw)),
    "scale_448_over_amax": ("quantize_rows", _scale_inverted),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTANTS))
def test_fp8_mutant_is_caught(name, monkeypatch):
    attr, fn = FP8_MUTANTS[name]
    monkeypatch.setattr(fp8, attr, fn)
    failed = []
    for pin in FP8_PINS:
        try:
            pin(fp8)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every FP8 pin"
