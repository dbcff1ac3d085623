"""The fused kernels' float-reciprocal quotient (`quot` in csrc/common.cuh)
restated in numpy float32, whose operations round the same way as the
device's: the correctly rounded reciprocal of b (`__frcp_rn`), the exact
conversion of a (`__int2float_rn`, a < 2^24), the round-to-nearest product
(`__fmul_rn`), truncation (`__float2int_rz`), then one correction step each
way. The kernels rely on it being exact for 0 <= a < 2^20 and 1 <= b < 2^14;
the cases that could break it are the ones next to a multiple of b, so every
a = n b - 1, n b, n b + 1 in range is checked for every b, plus every a below
4096 for the small divisors.
"""
import numpy as np

A_MAX = 1 << 20
B_MAX = 1 << 14


def quot(a: np.ndarray, b: int) -> np.ndarray:
    rb = np.float32(1.0) / np.float32(b)
    q = (a.astype(np.float32) * rb).astype(np.int64)     # float32 product, truncated
    r = a - q * b
    q += (r >= b).astype(np.int64)
    q -= (r < 0).astype(np.int64)
    return q


def test_quot_is_exact_next_to_every_multiple():
    for b in range(1, B_MAX):
        n = np.arange(0, A_MAX // b + 2, dtype=np.int64) * b
        a = np.concatenate([n - 1, n, n + 1])
        a = a[(a >= 0) & (a < A_MAX)]
        q = quot(a, b)
        bad = q != a // b
        assert not bad.any(), (b, a[bad][:4], q[bad][:4])


def test_quot_is_exact_for_small_divisors_everywhere_below_4096():
    a = np.arange(0, 4096, dtype=np.int64)
    for b in range(1, 256):
        assert np.array_equal(quot(a, b), a // b), b


def test_correction_steps_absorb_a_reciprocal_off_by_a_few_ulps():
    """In this range the truncated product alone is already exact; the two
    correction steps are the margin. With the reciprocal moved two float32
    ulps either way the plain truncation goes wrong next to some multiples,
    and the corrected quotient stays exact (the steps are not vacuous)."""
    plain_wrong = 0
    for b in (3, 7, 10, 13, 100, 528, 5000):
        a = np.arange(0, A_MAX, dtype=np.int64)
        rb0 = np.float32(1.0) / np.float32(b)
        for rb in (np.nextafter(np.nextafter(rb0, np.float32(0)), np.float32(0)),
                   np.nextafter(np.nextafter(rb0, np.float32(1)), np.float32(1))):
            q = (a.astype(np.float32) * rb).astype(np.int64)
            plain_wrong += int((q != a // b).sum())
            r = a - q * b
            q = q + (r >= b) - (r < 0)
            assert np.array_equal(q, a // b), b
    assert plain_wrong > 0
