"""The division-free E4M3 quantizer's method, emulated exactly on the CPU.

The GPU kernels form fl32(x / d) without a division by Markstein's
correction: y = RN(1/d), q = RN(x * y), then twice q = RN(q + RN(x - d*q) * y),
each residual and each correction a fused multiply-add.  This test re-runs that
sequence of fp32 operations exactly in numpy (every product of two fp32 values
is exact in fp64; the correction's sum is rounded to fp32 through TwoSum), and
checks that the codes it gives match the oracle's rule E4M3_RNE_sat(fl32(x / d))
for every bf16 pattern, over descales spread across the method's range
[2^-64, 2^64] and descales built to put quotients next to rounding boundaries.
It pins the method the kernels use; the GPU tests check the kernels
themselves against the oracle, bit for bit."""
import numpy as np

import oracle

_BITS = np.arange(65536, dtype=np.uint32)
with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
    _X = (_BITS << 16).view(np.float32).astype(np.float64)


def _rn32_sum(a32, b):
    """RN_fp32(a + b) for fp32 a and an fp64 b that holds its value exactly."""
    a = a32.astype(np.float64)
    with np.errstate(all="ignore"):
        s = a + b
        bb = s - a
        err = (a - (s - bb)) + (b - bb)  # TwoSum: s + err == a + b exactly
        s32 = s.astype(np.float32)
        up = s > s32.astype(np.float64)
        toward = np.where(up, np.float32(np.inf), np.float32(-np.inf)).astype(np.float32)
        nb = np.nextafter(s32, toward)
        mid = (s32.astype(np.float64) + nb.astype(np.float64)) / 2
        # s on the midpoint between s32 and its neighbour: the exact sum lies on err's side
        tie = (s == mid) & (err != 0) & np.isfinite(s)
        go = tie & (np.sign(err) == np.sign(nb.astype(np.float64) - s32.astype(np.float64)))
        return np.where(go, nb, s32).astype(np.float32)


def _method_codes(d):
    d32 = np.float32(d)
    y64 = np.float64(np.float32(1.0) / d32)  # RN(1/d): numpy's fp32 division is IEEE
    d64 = np.float64(d32)
    with np.errstate(all="ignore"):
        q = (_X * y64).astype(np.float32)
        for _ in range(2):
            r = (_X - d64 * q.astype(np.float64)).astype(np.float32)  # exact in fp64, one rounding
            q = _rn32_sum(q, r.astype(np.float64) * y64)
    code = oracle.e4m3_encode(q)
    flagged = (code & 0x7F) == 0x7F  # NaN code: the kernels take the IEEE division there
    code = (code & 0x7F) | ((_BITS >> 8) & 0x80).astype(np.uint8)  # the input's sign (d > 0)
    return code, flagged


def _descales():
    rng = np.random.default_rng(11)
    ds = [2.0 ** -64, 2.0 ** 64, 1.0, 5 / 64, 3 / 64, 0.75, 5.0, 35 / 448, 448.0]
    ds += list(2.0 ** rng.uniform(-64, 64, 60)) + list(10.0 ** rng.uniform(-4, 2, 60))
    ds += [np.ldexp(1 - 2.0 ** -24, e) for e in (-60, -20, -1, 0, 7, 40, 63)]
    ds += [np.ldexp(float((a << 20) + s), e - 23) for a in (8, 11, 15) for s in (-5, -1, 1, 7) for e in (-9, 0, 6)]
    ds += [m / 64 for m in range(1, 65)]
    return [float(np.float32(x)) for x in ds]


def test_division_free_quotient_method_matches_the_rule():
    total_flagged = 0
    for d in _descales():
        code, flagged = _method_codes(d)
        want = oracle.quantize_q(_BITS.astype(np.uint16), d)
        bad = np.nonzero((code != want) & ~flagged)[0]
        assert bad.size == 0, (d, [hex(int(b)) for b in bad[:5]])
        # flagged codes come only from NaN or infinite inputs or overflowing quotients
        x = _X[flagged]
        assert np.all(~np.isfinite(x) | (np.abs(x) / np.float64(np.float32(d)) > 3.0e38)), d
        total_flagged += int(flagged.sum())
    assert total_flagged > 0


def test_uncorrected_product_does_not_match_the_rule():
    """The pin has teeth: q = RN(x * RN(1/d)) alone, without the correction
    steps, rounds some quotients to the wrong code."""
    mism = 0
    for d in [np.ldexp(float((a << 20) + s), -23) for a in (8, 11, 15) for s in (-5, -1, 1, 7)]:
        d32 = np.float32(d)
        with np.errstate(all="ignore"):
            q = (_X * np.float64(np.float32(1.0) / d32)).astype(np.float32)
        code = oracle.e4m3_encode(q)
        want = oracle.quantize_q(_BITS.astype(np.uint16), float(d32))
        fin = np.isfinite(_X)
        mism += int(np.sum((code != want) & fin))
    assert mism > 0
