"""The engine's work-list divide, checked as a method on CPU.

The kernel divides small non-negative integers by runtime values with a
single-precision reciprocal estimate followed by one correction step (exact
below 2^21).  The hardware reciprocal is only known to within one ulp, so this
test models it as the correctly rounded reciprocal moved by -1, 0 and +1 ulp
and checks that the corrected quotient equals floor division in every case:
exhaustively over a < 2^21 for a set of divisors that includes the awkward ones
(1, powers of two and their neighbours, the SM count, values past 2^21 and 2^24),
and on random pairs.  It tests the arithmetic the kernel relies on, not the
compiled code (that is covered by the GPU parity tests, whose work lists all
go through it).
"""
import numpy as np
import pytest


def corrected_quotient(a, b, ulp_shift):
    a = np.asarray(a, np.int64)
    b = np.asarray(b, np.int64)
    rb = (np.float32(1.0) / b.astype(np.float32)).astype(np.float32)
    if ulp_shift:
        rb = np.nextafter(rb, np.float32(np.inf) if ulp_shift > 0 else np.float32(0)).astype(np.float32)
    t = (a.astype(np.float32) * rb).astype(np.float32)
    q = np.trunc(t).astype(np.int64)
    r = a - q * b
    return q + np.where(r >= b, 1, np.where(r < 0, -1, 0))


DIVISORS = [1, 2, 3, 5, 7, 9, 15, 16, 17, 31, 63, 64, 65, 127, 152, 153, 255, 304, 1023, 4095, 65535,
            (1 << 20) + 7, (1 << 21) - 1, (1 << 24) + 3]


@pytest.mark.parametrize("ulp_shift", [-1, 0, 1])
def test_exact_below_2_21_for_awkward_divisors(ulp_shift):
    a = np.arange(0, 1 << 21, dtype=np.int64)
    for b in DIVISORS:
        q = corrected_quotient(a, np.full_like(a, b), ulp_shift)
        assert np.array_equal(q, a // b), "divisor %d" % b


@pytest.mark.parametrize("ulp_shift", [-1, 0, 1])
def test_exact_on_random_pairs(ulp_shift):
    rng = np.random.default_rng(7)
    a = rng.integers(0, 1 << 21, 1_000_000)
    for hi in (300, 1 << 12, 1 << 22):
        b = rng.integers(1, hi, a.size)
        assert np.array_equal(corrected_quotient(a, b, ulp_shift), a // b)


def test_a_wrong_correction_is_caught():
    """Without the correction step the estimate alone is wrong somewhere in range (so the checks above
    can fail)."""
    a = np.arange(0, 1 << 21, dtype=np.int64)
    b = np.full_like(a, 3)
    rb = np.nextafter(np.float32(1.0) / np.float32(3), np.float32(0))
    q = np.trunc((a.astype(np.float32) * rb).astype(np.float32)).astype(np.int64)
    assert not np.array_equal(q, a // b)
