"""Pins for the oracle's numeric primitives: bf16 rounding, pow2_ceil, the e4m3 format and the fp8
round trip (deepseek_v41_ref::attn rustdoc page: pow2_ceil, act_quant_inplace, FP8_BLOCK = 32).

Each check is against something other than the oracle itself: torch's own bf16 and float8_e4m3fn
casts (library routines), the frexp/ldexp closed form of 2^ceil(log2 v), points of the E4M3 format
definition, hand-worked blocks, and the error bound of a 3-bit-mantissa round to nearest.
"""
import math

import numpy as np
import pytest
import torch


def _torch_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch_cast(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
        # exact halfway points between two bf16 values: ties go to even
        ((np.arange(0, 2000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)[1:],
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 65504.0, 1e-40, -1e-40], np.float32),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    assert np.array_equal(orc.f32_to_bf16(x), _torch_bf16_bits(x))
    assert np.array_equal(orc.bf16_to_f32(orc.f32_to_bf16(x)), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def _pow2_ceil_closed_form(v):
    m, e = math.frexp(float(v))  # v = m * 2^e, m in [0.5, 1)
    return float(v) if m == 0.5 else math.ldexp(1.0, e)


def test_pow2_ceil_closed_form(orc):
    rng = np.random.default_rng(2)
    v = np.abs(rng.standard_normal(5000).astype(np.float32)) * np.float32(10.0) ** rng.integers(-30, 30, 5000)
    v = v[(v > np.finfo(np.float32).tiny) & np.isfinite(v)].astype(np.float32)
    powers = np.ldexp(np.float32(1.0), np.arange(-120, 120)).astype(np.float32)
    just_above = np.nextafter(powers, np.float32(np.inf)).astype(np.float32)
    just_below = np.nextafter(powers, np.float32(0)).astype(np.float32)
    for arr in (v, powers, just_above, just_below[just_below > np.finfo(np.float32).tiny]):
        got = orc.pow2_ceil(arr)
        want = np.array([_pow2_ceil_closed_form(a) for a in arr], np.float32)
        assert np.array_equal(got, want)
    # the amax floor of the fp8 scale: 1e-4 / 448 lies between 2^-23 and 2^-22
    assert orc.pow2_ceil(np.float32(1e-4) / np.float32(448.0))[()] == np.float32(2.0 ** -22)


def test_e4m3_format_points(orc):
    # E4M3 ("fn"): bias 7, 3 mantissa bits, S.1111.111 = NaN, largest finite 1.75 * 2^8 = 448
    pts = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
           0x40: 2.0, 0x7E: 448.0, 0x78: 256.0, 0x80: -0.0, 0xFE: -448.0, 0xB8: -1.0}
    for code, val in pts.items():
        d = orc.e4m3_decode(np.array([code], np.uint8))[0]
        assert d == val and math.copysign(1, d) == math.copysign(1, val)
        assert orc.e4m3_encode(np.array([val], np.float32))[0] == code
    assert np.isnan(orc.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_table_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_encode_matches_torch_in_range(orc):
    # every finite bf16 value with |v| <= 448, plus random f32 values across the range
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint32) << 16
    v = allbits.view(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 448.0)]
    rng = np.random.default_rng(3)
    r = (rng.uniform(-1, 1, 200000) * 2.0 ** rng.integers(-12, 9, 200000)).astype(np.float32)
    r = r[np.abs(r) <= 448.0]
    for arr in (v, r):
        mine = orc.e4m3_encode(arr)
        ref = torch.from_numpy(arr).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(mine, ref)


def test_e4m3_encode_saturates(orc):
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38], np.float32)
    assert (orc.e4m3_encode(big) == 0x7E).all()
    assert (orc.e4m3_encode(-big) == 0xFE).all()


def _hand_block():
    """A block of 32 with its hand-worked round trip.  amax = 1.0, so s = pow2_ceil(1/448) = 2^-8
    (2^-9 < 1/448 < 2^-8) and v/s = 256 v.  On the e4m3 grid [64, 128) has quantum 8, [128, 256)
    quantum 16, [256, 512) quantum 32; subnormals have quantum 2^-9."""
    vals = np.zeros(32, np.float32)
    want_code = np.zeros(32, np.uint8)
    want_val = np.zeros(32, np.float32)
    rows = [
        (1.0, 0x78, 1.0),                 # 256 = 2^8 exactly: E = 8 -> biased 15, m = 0
        (0.30078125, 0x6A, 0.3125),       # bf16(0.3); 77 / 8 = 9.625 -> 10 -> 80 = (13 << 3 | 2)
        (-0.5, 0xF0, -0.5),               # -128: E = 7 -> biased 14, sign set
        (0.296875, 0x6A, 0.3125),         # 76 / 8 = 9.5, a tie -> even 10 -> 80
        (0.265625, 0x68, 0.25),           # 68 / 8 = 8.5, a tie -> even 8 -> 64
        (2.0 ** -15, 0x04, 2.0 ** -15),   # 2^-7: subnormal, 4 * 2^-9
        (3 * 2.0 ** -18, 0x02, 2.0 ** -16),  # 1.5 * 2^-9: tie -> even 2 -> 2^-8
        (2.0 ** -19, 0x00, 0.0),          # 2^-11: below half a quantum -> 0
        (-0.75, 0xF4, -0.75),             # -192 = -(8 + 4) * 16: E = 7, m = 4
    ]
    for i, (v, c, r) in enumerate(rows):
        vals[i], want_code[i], want_val[i] = v, c, r
    return vals, want_code, want_val


def test_act_quant_hand_block(orc):
    vals, want_code, want_val = _hand_block()
    bits = orc.f32_to_bf16(vals)
    assert np.array_equal(orc.bf16_to_f32(bits), vals)  # the inputs are bf16 values
    out, codes, se = orc.act_quant(bits[None, :])
    assert se[0, 0] == -8
    assert np.array_equal(codes[0], want_code)
    assert np.array_equal(orc.bf16_to_f32(out[0]), want_val)


def test_act_quant_special_blocks(orc):
    z = np.zeros((1, 64), np.uint16)
    out, codes, se = orc.act_quant(z)
    assert (codes == 0).all() and (out == 0).all() and (se == -22).all()  # amax floored at 1e-4
    x = np.zeros(32, np.float32)
    x[5] = 448.0
    x[6] = -3.0
    out, codes, se = orc.act_quant(orc.f32_to_bf16(x)[None])
    assert se[0, 0] == 0 and codes[0, 5] == 0x7E and orc.bf16_to_f32(out[0, 6]) == -3.0


def test_act_quant_properties_random(orc):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 512)).astype(np.float32) * (10.0 ** rng.integers(-6, 6, (64, 1)))
    x[3, :32] *= 1e-9  # a block far below the amax floor
    bits = orc.f32_to_bf16(x)
    xv = orc.bf16_to_f32(bits).reshape(64, 16, 32).astype(np.float64)
    out, codes, se = orc.act_quant(bits)
    outv = orc.bf16_to_f32(out).reshape(64, 16, 32).astype(np.float64)
    # scale exponent: the frexp closed form of pow2_ceil(max(amax, 1e-4) / 448) (f32 division)
    amax = np.abs(orc.bf16_to_f32(bits).reshape(64, 16, 32)).max(-1)
    q = (np.maximum(amax, np.float32(1e-4)) / np.float32(448.0)).astype(np.float32)
    want_se = np.array([[int(math.log2(_pow2_ceil_closed_form(v))) for v in row] for row in q])
    assert np.array_equal(se.astype(int), want_se)
    # the value is the decoded code times the power-of-two scale, exactly (bf16-exact round trip)
    dec = orc.e4m3_decode(codes).reshape(64, 16, 32).astype(np.float64)
    assert np.array_equal(outv, dec * np.ldexp(1.0, se.astype(int))[..., None])
    # codes agree with torch's float8_e4m3fn cast of v / s
    s = np.ldexp(np.float32(1.0), se.astype(int)).astype(np.float32)
    ratio = (orc.bf16_to_f32(bits).reshape(64, 16, 32) / s[..., None]).astype(np.float32)
    ratio = np.clip(ratio, -448, 448)
    ref = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes.reshape(64, 16, 32), ref)
    # error bound of round-to-nearest with 3 mantissa bits: half a quantum
    sc = np.ldexp(1.0, se.astype(int))[..., None]
    r = np.abs(xv) / sc
    quantum = np.where(r < 2.0 ** -6, 2.0 ** -9, np.ldexp(1.0, np.floor(np.log2(np.maximum(r, 1e-300))).astype(int) - 3))
    assert (np.abs(outv - xv) <= 0.5 * quantum * sc + 0.0).all()
    # idempotent
    out2, codes2, se2 = orc.act_quant(out)
    assert np.array_equal(out2, out)


# ------------------------------------------------------------------- fp8 weight storage (128 x 128 tiles)

def _fp8_case(seed, shape=(300, 260)):
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    from csa_inputs import fp8_weight
    return fp8_weight(shape, seed)


def test_fp8_weight_dequant_matches_torch(orc):
    """bf16(f32(e4m3(code) * tile scale)) against torch's own float8_e4m3fn decode, f32 product and bf16
    cast (library routines), on a ragged 300 x 260 matrix (tiles of 128: the last row and column of
    tiles are partial)."""
    codes, scales = _fp8_case(31)
    got = orc.dequant_fp8_blocks(codes, scales, 128)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
    full = torch.from_numpy(scales).repeat_interleave(128, 0).repeat_interleave(128, 1)[:300, :260]
    want = (t * full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_fp8_weight_dequant_power_of_two_scales_exact(orc):
    """With power-of-two tile scales nothing rounds: a 4-bit significand times 2^k is a bf16 value."""
    codes, _ = _fp8_case(32)
    k = np.array([[-12, -3, 0], [4, -7, 2], [1, -1, -9]], np.float64)
    scales = np.exp2(k).astype(np.float32)
    got = orc.bf16_to_f32(orc.dequant_fp8_blocks(codes, scales, 128)).astype(np.float64)
    full = np.repeat(np.repeat(k, 128, 0), 128, 1)[:300, :260]
    assert np.array_equal(got, orc.e4m3_decode(codes).astype(np.float64) * np.exp2(full))


def test_fp8_weight_dequant_tile_index(orc):
    """Doubling the scale of tile (row tile 1, column tile 2) changes exactly the nonzero codes of rows
    128..255 and columns 256..259, and nothing else (a transposed or shifted tile index fails)."""
    codes, scales = _fp8_case(33)
    s2 = scales.copy()
    s2[1, 2] *= 2
    d1 = orc.dequant_fp8_blocks(codes, scales, 128)
    d2 = orc.dequant_fp8_blocks(codes, s2, 128)
    changed = d1 != d2
    inside = np.zeros_like(changed)
    inside[128:256, 256:260] = True
    nonzero = (codes & 0x7F) != 0
    assert not (changed & ~inside).any()
    assert np.array_equal(changed[inside], nonzero[inside])
