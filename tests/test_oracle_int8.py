"""Pins for the oracle's int8 page quantiser (CPU only).

The rule (libmir-metal paged/mod.rs, KvPageFormat::Int8PerTokenHead and
write::quantized; the scale is absmax / 127 rounded to nearest-even) is
evaluated here a second, independent way: in exact rational arithmetic
(``fractions.Fraction``) with an explicit round-to-nearest-even onto binary32.
That fixes every code and scale bit by the IEEE-754 definition, without the
hardware divider or libm.  Hand-worked rows pin the tie rule, the zero row and
the case where dividing by the stored scale and multiplying by 127/amax give
different codes.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle_pools import bits

F32_MANT = 23
F32_EMIN = -126


def round_half_even(x: Fraction) -> int:
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def to_binary32(x: Fraction) -> Fraction:
    """Exact value of x rounded to the nearest binary32 (ties to even)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, F32_EMIN)
    step = Fraction(2) ** (e - F32_MANT)
    return sign * round_half_even(a / step) * step


def exact_quantize(row_f32):
    """Expected (codes, scale) of one row by the definition, in exact arithmetic."""
    xs = [Fraction(float(v)) for v in row_f32]
    amax = max(abs(v) for v in xs)
    scale = to_binary32(amax / 127)
    if amax == 0:
        return [0] * len(xs), 0.0
    codes = []
    for v in xs:
        qt = to_binary32(v / scale)
        c = round_half_even(qt)
        codes.append(max(-127, min(127, c)))
    return codes, float(scale)


def _bf16(vals, d):
    row = torch.zeros(d, dtype=torch.float32)
    row[:len(vals)] = torch.tensor(vals, dtype=torch.float32)
    out = row.to(torch.bfloat16)
    assert torch.equal(out.float(), row), "hand-worked values must be exact in bf16"
    return out


def _quantize(rows: torch.Tensor):
    """Quantise rows [n, D] (bf16) through the oracle's write with one kv head."""
    n, D = rows.shape
    dims = oracle.Dims(n, 1, 1, D)
    kp = np.zeros(dims.pool_shape, np.int8)
    vp = np.zeros(dims.pool_shape, np.int8)
    ks = np.zeros(dims.scale_shape, np.float32)
    vs = np.zeros(dims.scale_shape, np.float32)
    table = np.arange(n, dtype=np.int32)[None]
    k = rows.view(1, n, 1, D)
    st = oracle.write_int8(k, -k, kp, vp, ks, vs, dims, table, np.zeros(1, np.int32))
    assert st == oracle.OK
    return kp[:n, 0, 0], ks[:n, 0, 0], vp[:n, 0, 0], vs[:n, 0, 0]


# (row values, expected leading codes, expected scale) -- worked by hand:
HAND_ROWS = [
    # amax 127 -> scale exactly 1; 63.5 and 0.5 are ties: to even -> 64 and 0
    ([127.0, 63.5, -1.0, 0.5, -0.5, 1.5, 2.5], [127, 64, -1, 0, 0, 2, 2], 1.0),
    # amax 254 -> scale exactly 2; 5/2 = 2.5 -> 2, 7/2 = 3.5 -> 4, -3/2 -> -2
    ([-254.0, 5.0, 7.0, -3.0, 1.0], [-127, 2, 4, -2, 0], 2.0),
    # all zeros: scale 0, codes 0
    ([], [0, 0, 0], 0.0),
    # a negative absmax maps to -127; 63.5 ties to 64 after the exact /1
    ([-127.0, 63.5, 62.5], [-127, 64, 62], 1.0),
]


@pytest.mark.parametrize("vals,codes,scale", HAND_ROWS)
def test_hand_worked_rows(vals, codes, scale):
    D = 16
    c, s, cv, sv = _quantize(_bf16(vals, D)[None])
    assert s[0] == np.float32(scale)
    assert list(c[0, :len(codes)]) == codes
    assert (c[0, max(len(vals), len(codes)):] == 0).all()
    # V was written negated: symmetric rule
    assert sv[0] == s[0] and np.array_equal(cv[0], -c[0])


def test_division_by_stored_scale_not_reciprocal_multiply():
    """amax = 1.59375, x = amax / 2: fl32(amax/127) = 0.0125492122...,
    x / scale rounds to 63.500004 -> 64, while x * fl32(127/amax) = 63.499996
    would give 63.  amax = 1.6171875 is the opposite case (63 by division).
    2.96875 / 2 lands exactly on 63.5 in binary32 and ties to 64."""
    cases = [(1.59375, 0.796875, 64), (1.6171875, 0.80859375, 63), (2.96875, 1.484375, 64),
             (0.77734375, -0.388671875, -64), (0.578125, -0.2890625, -63)]
    rows = torch.stack([_bf16([a, x], 8) for a, x, _ in cases])
    c, s, _, _ = _quantize(rows)
    for i, (a, x, want) in enumerate(cases):
        codes, scale = exact_quantize(rows[i].float().numpy())
        assert codes[1] == want, "hand value disagrees with exact arithmetic"
        assert c[i, 1] == want and c[i, 0] == 127
        assert s[i] == np.float32(scale)


@pytest.mark.parametrize("D,seed", [(64, 0), (128, 1), (8, 2)])
def test_random_rows_equal_exact_rational_rule(D, seed):
    g = torch.Generator().manual_seed(seed)
    n = 96
    rows = (torch.randn((n, D), generator=g) *
            torch.exp(torch.randn((n, 1), generator=g) * 3)).to(torch.bfloat16)
    rows[0] = 0
    rows[1, :] = rows[1, 0]  # constant row: every code is +-127
    c, s, _, _ = _quantize(rows)
    for i in range(n):
        codes, scale = exact_quantize(rows[i].float().numpy())
        assert s[i] == np.float32(scale), i
        assert list(c[i]) == codes, i


def test_quantiser_properties():
    g = torch.Generator().manual_seed(9)
    rows = torch.randn((200, 128), generator=g).to(torch.bfloat16)
    c, s, _, _ = _quantize(rows)
    x = rows.float().numpy()
    amax = np.abs(x).max(axis=1)
    assert (np.abs(c.astype(np.int32)) <= 127).all()
    # the absmax element maps to +-127 with the sign of x
    arg = np.abs(x).argmax(axis=1)
    assert (c[np.arange(200), arg] == np.sign(x[np.arange(200), arg]) * 127).all()
    # reconstruction error at most half a step (plus binary32 rounding of the quotient)
    err = np.abs(x - c.astype(np.float64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None] * (0.5 + 2.0 ** -16)).all()
    # power-of-two rescaling commutes with the rule: codes equal, scale doubles
    c2, s2, _, _ = _quantize((rows.float() * 2).to(torch.bfloat16))
    assert np.array_equal(c2, c) and np.array_equal(s2, s * 2)


def test_int8_write_uses_the_same_slot_map():
    """Quantised pages sit where native pages would (identity table: storage order)."""
    g = torch.Generator().manual_seed(5)
    bs, hkv, D, L = 4, 2, 16, 11
    nb = 4
    dims = oracle.Dims(nb, bs, hkv, D)
    k = torch.randn((1, L, hkv, D), generator=g).to(torch.bfloat16)
    kp = np.full(dims.pool_shape, 99, np.int8)
    vp = kp.copy()
    ks = np.full(dims.scale_shape, -1, np.float32)
    vs = ks.copy()
    table = np.arange(nb, dtype=np.int32)[None]
    assert oracle.write_int8(k, k, kp, vp, ks, vs, dims, table, np.zeros(1, np.int32)) == 0
    flat = kp.reshape(-1, hkv, D)
    fs = ks.reshape(-1, hkv)
    for t in range(L):
        for h in range(hkv):
            codes, scale = exact_quantize(k[0, t, h].float().numpy())
            assert list(flat[t, h]) == codes and fs[t, h] == np.float32(scale)
    assert (flat[L:] == 99).all() and (fs[L:] == -1).all()
