"""Host logic of the stack-step check (tests/helpers.py check_rmsnorm_bf16), on the CPU.

The GPU test of the residual RMS-norm stack step allows exactly one kind of difference
from the oracle: a 1-ulp bf16 difference where the exact normalised value sits at a bf16
rounding tie.  These cases pin that rule: equal bits pass, a 1-ulp flip away from a tie
fails, a flip at a tie passes and is counted, a 2-ulp or sign difference fails."""
import numpy as np
import pytest

from oracle import oracle as O
from tests.helpers import check_rmsnorm_bf16


def _row():
    return np.random.default_rng(12).normal(size=(2, 512)).astype(np.float32)


def test_equal_bits_pass():
    x = _row()
    assert check_rmsnorm_bf16(x, O.rmsnorm_bf16(x.astype(np.float64))) == 0


def test_flip_away_from_a_tie_fails():
    x = _row()
    xn = O.rmsnorm_bf16(x.astype(np.float64)).copy()
    xn[0, 3] += 1
    with pytest.raises(AssertionError):
        check_rmsnorm_bf16(x, xn)


@pytest.mark.parametrize("delta", [2, 0x8000])
def test_two_ulp_or_sign_difference_fails(delta):
    x = _row()
    xn = O.rmsnorm_bf16(x.astype(np.float64)).copy()
    xn[1, 7] ^= delta if delta == 0x8000 else 0
    if delta == 2:
        xn[1, 7] += 2
    with pytest.raises(AssertionError):
        check_rmsnorm_bf16(x, xn)


def test_flip_at_a_tie_passes_and_is_counted():
    # 64 entries of 1.0 and one of v: mean square m = (64 + v^2) / 65; choose the entry so
    # that v / sqrt(m) is (to fp64 precision) the midpoint 1 + 2^-8 of the bf16 values 1 and
    # 1 + 2^-7; either rounding is then allowed
    t = 1.0 + 2.0 ** -8
    # v / sqrt((64 + v^2) / 65) = t  =>  v^2 (65 - t^2) = 64 t^2
    v = np.sqrt(64 * t * t / (65 - t * t))
    x = np.ones((1, 65))
    x[0, 0] = v
    x32 = x.astype(np.float32)
    ref = O.rmsnorm_bf16(x32.astype(np.float64), eps=0.0)
    other = ref.copy()
    other[0, 0] = 0x3F80 if ref[0, 0] == 0x3F81 else 0x3F81
    assert {int(ref[0, 0]), int(other[0, 0])} == {0x3F80, 0x3F81}
    assert check_rmsnorm_bf16(x32, other, eps=0.0) == 1
