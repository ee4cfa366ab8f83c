"""Pins for the 8-bit cache oracle: E4M3 codes against a library routine (PyTorch's float8_e4m3fn casts) and
the format's closed forms, the row exponent against its defining inequality, the quantizer against brute
force over all codes, and planted mistakes that each pin must catch."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8


def _torch_decode_all():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _torch_encode(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_table_matches_library():
    ours, lib = fp8.e4m3_table(), _torch_decode_all()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[~np.isnan(ours)], lib[~np.isnan(lib)])


def test_decode_closed_forms():
    """The E4M3 layout: bias 7, subnormals at exponent field 0, S.1111.111 the only NaNs, no infinities."""
    assert fp8.e4m3_decode(0x7E) == 448.0                  # largest finite
    assert fp8.e4m3_decode(0x08) == 2.0 ** -6              # smallest normal
    assert fp8.e4m3_decode(0x01) == 2.0 ** -9              # smallest subnormal
    assert fp8.e4m3_decode(0x07) == 7 * 2.0 ** -9          # largest subnormal
    assert fp8.e4m3_decode(0x38) == 1.0
    assert fp8.e4m3_decode(0x39) == 1.125
    assert fp8.e4m3_decode(0xB8) == -1.0
    assert fp8.e4m3_decode(0x80) == 0.0 and math.copysign(1.0, fp8.e4m3_decode(0x80)) < 0
    nans = [c for c in range(256) if math.isnan(fp8.e4m3_decode(c))]
    assert nans == [0x7F, 0xFF]
    finite = sorted(fp8.e4m3_decode(c) for c in range(0x7F))
    assert len(set(finite)) == 127 and all(np.diff(finite) > 0)


def test_encode_matches_library_on_codes_midpoints_and_random():
    vals = [v for v, _ in fp8._finite_codes()]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]        # exact ties: even code wins
    rng = np.random.default_rng(0)
    rnd = list(rng.uniform(-448, 448, 400)) + list(rng.standard_normal(400) * 0.01)
    xs = np.array(vals + mids + [-m for m in mids] + rnd, dtype=np.float32)
    assert np.all(xs.astype(np.float64) == np.array(vals + mids + [-m for m in mids] + rnd, dtype=np.float64)
                  .astype(np.float32).astype(np.float64))
    ours = np.array([fp8.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(ours, _torch_encode(xs))


def test_array_encoder_matches_scalar_definition():
    vals = [v for v, _ in fp8._finite_codes()]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    rng = np.random.default_rng(5)
    y = np.array(vals + mids + [-m for m in mids] + list(rng.uniform(-448, 448, 500)) + [0.0, -0.0])
    assert np.array_equal(fp8.e4m3_encode_array(y), np.array([fp8.e4m3_encode(v) for v in y], dtype=np.uint8))
    amax = np.concatenate([np.exp2(rng.uniform(-24, 16, 500)), [0.0, 448.0, 449.0, 224.0, 224.125, 65504.0]])
    amax = amax.astype(np.float16).astype(np.float64)
    assert list(fp8.row_exponents(amax)) == [fp8.row_exponent(a) for a in amax]
    x = _rows(rng, 6, 32)
    c1, s1 = fp8.quantize_rows(x)
    for i in range(6):
        c2, s2 = fp8.quantize_row(x[i])
        assert np.array_equal(c1[i], c2) and s1[i] == s2


def test_encode_ties_go_to_even():
    assert fp8.e4m3_encode(1.0625) == 0x38    # between 1.0 (m=0) and 1.125 (m=1)
    assert fp8.e4m3_encode(1.1875) == 0x3A    # between 1.125 (m=1) and 1.25 (m=2)
    assert fp8.e4m3_encode(2.0 ** -10) == 0x00  # between 0 and the smallest subnormal
    assert fp8.e4m3_encode(3 * 2.0 ** -10) == 0x02
    assert fp8.e4m3_encode(432.0) == 0x7E     # between 416 (m=5) and 448 (m=6): 448 has the even mantissa


@pytest.mark.parametrize("amax,e", [(0.0, 0), (448.0, 0), (449.0, 1), (224.0, -1), (224.125, 0), (1.0, -8),
                                    (1.75, -8), (1.7509765625, -7), (65504.0, 8), (2.0 ** -24, -32)])
def test_row_exponent_values(amax, e):
    assert fp8.row_exponent(amax) == e


def test_row_exponent_defining_inequality():
    rng = np.random.default_rng(1)
    for a in np.concatenate([rng.uniform(0, 65504, 300), np.exp2(rng.uniform(-24, 16, 300))]):
        a = float(np.float16(a))
        if a == 0:
            continue
        e = fp8.row_exponent(a)
        assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)
        assert e == math.ceil(math.log2(a / 448.0)) or a / 448.0 == 2.0 ** e


def _rows(rng, n, d):
    mags = np.exp2(rng.uniform(-12, 12, size=(n, 1)))
    return (rng.standard_normal((n, d)) * mags).astype(np.float16)


def test_quantize_row_is_nearest_grid_point_brute_force():
    rng = np.random.default_rng(2)
    table = fp8.e4m3_table()
    finite = ~np.isnan(table)
    for x in _rows(rng, 12, 16):
        codes, sb = fp8.quantize_row(x)
        e = sb - fp8.SCALE_BIAS
        grid = table[finite] * 2.0 ** e
        for xi, c in zip(x.astype(np.float64), codes):
            got = table[c] * 2.0 ** e
            best = np.min(np.abs(grid - xi))
            assert abs(got - xi) == best
        assert np.max(np.abs(table[codes])) > 224.0 or np.all(x == 0)


def test_quantize_error_bound_and_fp16_exactness():
    rng = np.random.default_rng(3)
    x = _rows(rng, 64, 128)
    codes, scales = fp8.quantize_rows(x)
    xh = fp8.dequantize_rows(codes, scales)
    xf = x.astype(np.float64)
    e = (scales.astype(np.float64) - 127)[:, None]
    eb = np.broadcast_to(e, xf.shape)
    err = np.abs(xh - xf)
    normal = np.abs(xf) >= 2.0 ** (eb - 6)                 # x / 2^e in the normal range of E4M3
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf)[normal])   # half an ulp of a 3-bit mantissa
    assert np.all(err[~normal] <= 2.0 ** (eb[~normal] - 10))       # half the subnormal spacing 2^-9
    # every dequantized value is an fp16 value (the kernels rely on this for exact dequantization)
    assert np.array_equal(xh.astype(np.float16).astype(np.float64), xh)


def test_zero_row_and_sign():
    codes, sb = fp8.quantize_row(np.zeros(8, dtype=np.float16))
    assert sb == 127 and np.all(codes == 0)
    codes, sb = fp8.quantize_row(np.array([-448, 448, -1, 0], dtype=np.float16))
    assert sb == 127 and list(codes) == [0xFE, 0x7E, 0xB8, 0x00]


def test_append_reference_8bit_brute_force():
    rng = np.random.default_rng(4)
    nb, hkv, bs, d = 5, 2, 16, 8
    ck = np.zeros((nb, hkv, bs, d), np.uint8)
    cv = np.zeros_like(ck)
    sc = np.zeros((nb, hkv, 2, bs), np.uint8)
    k = _rows(rng, 3 * hkv, d).reshape(3, hkv, d)
    v = _rows(rng, 3 * hkv, d).reshape(3, hkv, d)
    slots = [17, -1, 79]
    fp8.append_reference_8bit(ck, cv, sc, k, v, slots)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(hkv):
            c, b = fp8.quantize_row(k[t, h])
            assert np.array_equal(ck[s // bs, h, s % bs], c) and sc[s // bs, h, 0, s % bs] == b
            c, b = fp8.quantize_row(v[t, h])
            assert np.array_equal(cv[s // bs, h, s % bs], c) and sc[s // bs, h, 1, s % bs] == b
    touched = {(s // bs, s % bs) for s in slots if s >= 0}
    for blk in range(nb):
        for off in range(bs):
            if (blk, off) not in touched:
                assert not ck[blk, :, off].any() and not sc[blk, :, :, off].any()


# ---- planted mistakes: each variant of the quantizer must fail one of the checks above ----

def _mutant_decode(kind):
    def dec(code):
        sign = -1.0 if code & 0x80 else 1.0
        exp, man = (code >> 3) & 0xF, code & 7
        bias = 8 if kind == "bias8" else 7
        if exp == 0xF and man == 7:
            return math.nan
        if exp == 0:
            lead = 1.0 if kind == "no_subnormal" else 0.0
            return sign * (lead + man / 8.0) * 2.0 ** (1 - bias)
        return sign * (1.0 + man / 8.0) * 2.0 ** (exp - bias)
    return dec


@pytest.mark.parametrize("kind", ["bias8", "no_subnormal"])
def test_decode_mutants_are_caught(kind):
    dec = _mutant_decode(kind)
    table = np.array([dec(c) for c in range(256)])
    lib = _torch_decode_all()
    ok = np.array_equal(np.isnan(table), np.isnan(lib)) and np.array_equal(table[~np.isnan(table)], lib[~np.isnan(lib)])
    assert not ok


@pytest.mark.parametrize("kind", ["truncate", "ties_away", "exponent_floor"])
def test_quantizer_mutants_are_caught(kind):
    table = fp8.e4m3_table()

    def enc(x):
        a = abs(x)
        vals = [(v, c) for v, c in fp8._finite_codes()]
        if kind == "truncate":
            c = max(c for v, c in vals if v <= a)
        else:
            c = min(vals, key=lambda vc: (abs(a - vc[0]), -vc[0] if kind == "ties_away" else vc[1] & 1))[1]
        return (0x80 if x < 0 else 0) | c

    def row_exp(a):
        if kind != "exponent_floor" or a == 0:
            return fp8.row_exponent(a)
        return math.floor(math.log2(a / 448.0))

    caught = False
    vals = [v for v, _ in fp8._finite_codes()]
    mids = np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])] + [3.3, 100.7], dtype=np.float32)
    if not np.array_equal(np.array([enc(float(m)) for m in mids], np.uint8), _torch_encode(mids)):
        caught = True
    for a in [449.0, 224.125, 1000.0]:
        e = row_exp(a)
        if not (a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)):
            caught = True
    assert caught, kind


def test_quantizing_twice_changes_nothing():
    """Dequantized rows are fixed points: quantizing them again gives back the same values.  (Not always the
    same codes and scale: a row whose largest value rounded down to 224 * 2^e is stored again as 448 * 2^(e-1).)"""
    rng = np.random.default_rng(6)
    x = _rows(rng, 40, 64)
    xh = fp8.dequantize_rows(*fp8.quantize_rows(x))
    xh2 = fp8.dequantize_rows(*fp8.quantize_rows(xh.astype(np.float16)))
    assert np.array_equal(xh, xh2)


def test_values_on_the_grid_come_back_exactly():
    """A row built from E4M3 values times 2^e (its largest magnitude in (224, 448] * 2^e) is stored exactly."""
    rng = np.random.default_rng(7)
    table = fp8.e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])])
    for e in (-15, -8, 0, 5):     # from 2^-15 on, every E4M3 value times 2^e is an fp16 number
        codes = rng.choice(finite, size=32)
        codes[3] = 0x7E                                   # 448: the row's largest magnitude
        x = (table[codes] * 2.0 ** e).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), table[codes] * 2.0 ** e)
        c, sb = fp8.quantize_row(x)
        assert sb - fp8.SCALE_BIAS == e
        assert np.array_equal(fp8.dequantize_row(c, sb), x.astype(np.float64))


def test_only_the_top_of_the_fp16_range_dequantizes_past_it():
    """The reading behind the 8-bit prefill shadow: a dequantized value leaves the fp16 range only when the
    row's exponent is 8 and the value rounds up to 256 * 2^8 = 65536, i.e. |x| >= 63488 (within 3 % of the
    fp16 maximum 65504)."""
    c, sb = fp8.quantize_row(np.array([63488.0, 1.0], dtype=np.float16))
    assert sb - fp8.SCALE_BIAS == 8 and fp8.dequantize_row(c, sb)[0] == 65536.0
    c, sb = fp8.quantize_row(np.array([63456.0, 1.0], dtype=np.float16))   # the fp16 value just below
    assert fp8.dequantize_row(c, sb)[0] == 61440.0
    rng = np.random.default_rng(8)
    x = (rng.uniform(-1, 1, size=(200, 64)) * np.exp2(rng.uniform(-24, 15.9, size=(200, 1)))).astype(np.float16)
    x = x[np.abs(x.astype(np.float64)).max(axis=1) < 63488]
    xh = fp8.dequantize_rows(*fp8.quantize_rows(x))
    assert np.abs(xh).max() <= 65504 and np.array_equal(xh.astype(np.float16).astype(np.float64), xh)
