"""The int8 page write finds each code without a division per element: it
multiplies by the correctly rounded reciprocal of the scale and falls back
to the IEEE division only when the product lies within 3e-5 of a
half-integer.  The bound behind it: fl(x * fl(1/scale)) is within
|x/scale| * (2^-23 + 2^-48) <= 1.53e-5 of x/scale for |x/scale| < 128, and
fl(x/scale) within half an ulp (<= 3.8e-6).  Checked here in numpy binary32
(IEEE division and multiplication) over every pair of positive bf16 values
(amax, x <= amax) in [2^-3, 2^3): each pair where the two rint() differ lies
inside the band.  CPU only; the GPU parity of the write itself is in
test_gpu_parity.py."""
import numpy as np

BAND = np.float32(3e-5)


def bf16_values(lo_bits, hi_bits):
    u = np.arange(lo_bits, hi_bits, dtype=np.uint32)
    return (u << 16).view(np.float32)


def test_every_disagreement_lies_in_the_division_band():
    vals = bf16_values(0x3e00, 0x4100)              # 0.125 .. 8 (exclusive)
    n_band = n_diff = n_pairs = 0
    for amax in vals:
        scale = np.float32(amax) / np.float32(127)
        rcp = np.float32(1) / scale
        xs = vals[vals <= amax]
        xs = np.concatenate([xs, -xs])
        exact = xs / scale
        fast = xs * rcp
        frac = fast - np.floor(fast)
        band = np.abs(frac - np.float32(0.5)) <= BAND
        diff = np.rint(exact) != np.rint(fast)
        assert not (diff & ~band).any(), amax
        n_band += int(band.sum())
        n_pairs += len(xs)
        n_diff += int(diff.sum())
    # the band is rare (bf16 pairs are structured: x = amax / 2 lands near
    # 63.5), and the disagreements it catches are real
    assert n_diff > 0 and n_band < 0.01 * n_pairs
