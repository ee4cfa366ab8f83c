"""8-bit cache oracle: FP8 E4M3 codes with one power-of-two scale per cached (token, KV head) row.

Test infrastructure only (see the package docstring).

What the pages fix: when the cache is the binding limit, quantize it ("Continuous Batching Is Not a Bigger
Batch", section "Checking it on a real system"); an 8-bit cache holds half the raw bytes of an fp16 one, with
scales on top ("An advertised batch limit proves nothing until sampled", section "Context math sets the
ceiling the fields ignore").  They fix neither the 8-bit format nor the scale granularity.  Readings taken
(each listed in the design notes):

  * codes are FP8 E4M3 as the OCP 8-bit floating point specification defines it (1 sign bit, 4 exponent
    bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN; no infinities;
    largest finite magnitude 448);
  * one scale per cached row -- a token's d values of one KV head, K and V separately -- so appending a
    token never touches another token's codes;
  * the scale is a power of two 2^e, stored as the byte e + 127 (the E8M0 scale encoding of the OCP
    microscaling formats), with e the smallest integer such that the row's largest magnitude is at most
    448 * 2^e (e = 0 for an all-zero row); no value is clipped;
  * codes are the E4M3 value nearest to x / 2^e, ties to the even code (IEEE round-to-nearest-even);
  * attention reads the dequantized values code * 2^e exactly.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
SCALE_BIAS = 127


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte (OCP 8-bit floating point specification, E4M3 encoding)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)          # subnormal: 0.mmm x 2^(1 - bias)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


def e4m3_table() -> np.ndarray:
    """float64 [256]: the value of every code, index = code."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def _finite_codes() -> list[tuple[float, int]]:
    """(value, code) of every non-negative finite code, ascending (0x00 .. 0x7E)."""
    return [(e4m3_decode(c), c) for c in range(0x7F)]


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code to x, ties to the code with an even mantissa; |x| above 448 saturates to +-448
    (never reached by the row quantizer below); NaN gives 0x7F.  By search over the 127 non-negative finite
    codes: slow and plainly the definition."""
    x = float(x)
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0x00
    a = abs(x)
    best_val, best_code = None, None
    for val, code in _finite_codes():
        if best_code is None:
            best_val, best_code = val, code
            continue
        d_new, d_best = abs(a - val), abs(a - best_val)
        if d_new < d_best or (d_new == d_best and (code & 1) == 0 and (best_code & 1) == 1):
            best_val, best_code = val, code
    return sign | best_code


def e4m3_encode_array(y: np.ndarray) -> np.ndarray:
    """e4m3_encode on every element of a finite float64 array with |y| <= 448: the same nearest-code rule
    evaluated for many values at once.  A search of the ascending code values brackets |y| between two
    neighbours; the nearer one wins, the even code on a tie."""
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)) and np.all(np.abs(y) <= E4M3_MAX)
    vals = np.array([v for v, _ in _finite_codes()], dtype=np.float64)   # code c has value vals[c]
    a = np.abs(y)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)  # vals[hi] >= a (first such)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(a == vals[hi], hi, code)
    return (code | (np.signbit(y).astype(np.int64) << 7)).astype(np.uint8)


def row_exponents(amax: np.ndarray) -> np.ndarray:
    """row_exponent of every element: a first guess from log2, then exact corrections by the defining
    inequality (448 * 2^(e-1) < amax <= 448 * 2^e), all comparisons exact in float64."""
    amax = np.asarray(amax, dtype=np.float64)
    assert np.all(amax >= 0) and np.all(np.isfinite(amax))
    pos = amax > 0
    e = np.zeros(amax.shape, dtype=np.int64)
    e[pos] = np.ceil(np.log2(amax[pos] / E4M3_MAX)).astype(np.int64)
    for _ in range(4):
        up = pos & (amax > E4M3_MAX * np.exp2(e.astype(np.float64)))
        down = pos & (amax <= E4M3_MAX * np.exp2((e - 1).astype(np.float64)))
        e = e + up.astype(np.int64) - down.astype(np.int64)
    assert not np.any(pos & ((amax > E4M3_MAX * np.exp2(e.astype(np.float64))) |
                             (amax <= E4M3_MAX * np.exp2((e - 1).astype(np.float64)))))
    return e


def row_exponent(amax: float) -> int:
    """Smallest integer e with amax <= 448 * 2^e (0 for amax == 0).  Comparisons are exact in float64."""
    amax = float(amax)
    assert amax >= 0 and math.isfinite(amax)
    if amax == 0.0:
        return 0
    e = 0
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    while amax <= E4M3_MAX * 2.0 ** (e - 1):
        e -= 1
    return e


def quantize_row(x: np.ndarray) -> tuple[np.ndarray, int]:
    """One cached row (fp16 [d]) -> (uint8 codes [d], scale byte e + 127)."""
    xf = np.asarray(x, dtype=np.float64)
    assert np.all(np.isfinite(xf)), "the 8-bit cache takes finite keys and values"
    e = row_exponent(float(np.max(np.abs(xf))) if xf.size else 0.0)
    codes = np.array([e4m3_encode(v / 2.0 ** e) for v in xf], dtype=np.uint8)
    return codes, e + SCALE_BIAS


def dequantize_row(codes: np.ndarray, scale_byte: int) -> np.ndarray:
    """float64 [d]: code value x 2^(scale_byte - 127)."""
    table = e4m3_table()
    return table[np.asarray(codes, dtype=np.int64)] * 2.0 ** (int(scale_byte) - SCALE_BIAS)


def quantize_rows(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp16 [..., d] -> (uint8 codes [..., d], uint8 scale bytes [...]): quantize_row on every row, with the
    exponents from row_exponents and the codes from e4m3_encode_array."""
    x = np.asarray(x)
    flat = x.reshape(-1, x.shape[-1]).astype(np.float64)
    assert np.all(np.isfinite(flat)), "the 8-bit cache takes finite keys and values"
    exps = row_exponents(np.max(np.abs(flat), axis=1) if flat.shape[1] else np.zeros(flat.shape[0]))
    codes = e4m3_encode_array(flat / np.exp2(exps.astype(np.float64))[:, None])
    return codes.reshape(x.shape), (exps + SCALE_BIAS).astype(np.uint8).reshape(x.shape[:-1])


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 [..., d] from codes [..., d] and scale bytes [...]."""
    table = e4m3_table()
    exps = np.asarray(scales, dtype=np.float64) - SCALE_BIAS
    return table[np.asarray(codes, dtype=np.int64)] * np.exp2(exps)[..., None]


def append_reference_8bit(codes_k: np.ndarray, codes_v: np.ndarray, scales: np.ndarray, k: np.ndarray,
                          v: np.ndarray, slot_mapping) -> None:
    """In place, one layer of an 8-bit pool: the new tokens' rows quantized into their slots.

    codes_k, codes_v: uint8 [num_blocks, Hkv, bs, d]; scales: uint8 [num_blocks, Hkv, 2 (K, V), bs];
    k, v: fp16 [T, Hkv, d].  Slot -1 is skipped ("Continuous Batching Is Not a Bigger Batch", opening section
    and "The allocator is the other half": every computed token's key and value are stored in its slot).
    """
    block_size = codes_k.shape[2]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        for h in range(k.shape[1]):
            codes_k[blk, h, off], scales[blk, h, 0, off] = quantize_row(k[t, h])
            codes_v[blk, h, off], scales[blk, h, 1, off] = quantize_row(v[t, h])
